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
