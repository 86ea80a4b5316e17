"""Host logic of bench.py that needs no GPU: which linears of a step share a launch group."""
import bench


def _names(layers, linears):
    return [f"L{l}.{name}" for l in range(layers) for name, _, _ in linears]


def test_decoder_layer_groups():
    # q, k, v read the same input; so do gate and up; o and down each follow the linear before them
    names = _names(2, bench._L8)
    assert bench.launch_groups(names) == [[0, 1, 2], [3], [4, 5], [6], [7, 8, 9], [10], [11, 12], [13]]
    assert [len(g) for g in bench.launch_groups(_names(8, bench._L70))] == [3, 1, 2, 1] * 8


def test_unrelated_linears_stay_in_order():
    for wl in ("sweep-int4a", "int8s-8192", "int2a-8192", "nf4-8192"):
        spec = bench.WORKLOADS[wl]
        names = _names(3, spec["linears"])
        assert bench.launch_groups(names) == [[i] for i in range(len(names))]


def test_groups_cover_every_linear_once():
    names = _names(4, bench._L8)
    flat = [i for g in bench.launch_groups(names) for i in g]
    assert flat == list(range(len(names)))


def _recs(layers, linears):
    return [dict(name=f"L{l}.{name}", N=n, K=k) for l in range(layers) for name, n, k in linears]


def test_gate_and_up_pair_into_one_op():
    ops = bench.step_ops(_recs(2, bench._L8), gated=True)
    assert [op["kind"] for op in ops] == ["gemm"] * 4 + ["gated", "gemm"] + ["gemm"] * 4 + ["gated", "gemm"]
    assert ops[4]["name"] == "L0.gate_up" and [r["name"] for r in ops[4]["recs"]] == ["L0.gate", "L0.up"]
    # q, k, v still share a launch group; the gated op and down each stand alone
    assert bench.launch_groups([op["name"] for op in ops])[:4] == [[0, 1, 2], [3], [4], [5]]
    assert [op["kind"] for op in bench.step_ops(_recs(2, bench._L8), gated=False)] == ["gemm"] * 14


def test_gated_bytes_count_x_and_h_once():
    fmt, g, N, K, M = "INT4_ASYM", 128, 14336, 4096, 1
    both = 2 * bench.alg_bytes(fmt, g, N, K, M)
    assert bench.gated_bytes(fmt, g, N, K, M) == both - 2 * M * K - 2 * M * N
