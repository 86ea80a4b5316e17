"""Host logic of bench.py that needs no GPU: which linears of a step share a launch group, the
profile fields the bench line reads, the dominant kernel's name and the roofline time."""
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


def _fake_tree(tmp_path, sha, ratio="1.0015", share="0.912"):
    csrc = tmp_path / "gemm_uq_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "uq_gemv.cuh").write_text("kernel a\n")
    (csrc / "uq_common.cuh").write_text("kernel b\n")
    (csrc / "uq_tc.cu").write_text("not hashed\n")
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "gemv_w.md").write_text(f"# summary\n\n- kernel_source_sha: {sha}\n- dram_over_algorithmic: {ratio}\n")
    (prof / "launches_w.md").write_text(f"# launches\n\n- dominant_share: {share}\n")
    return tmp_path


def test_traffic_only_from_a_profile_of_the_current_sources(tmp_path, monkeypatch):
    root = _fake_tree(tmp_path, "0" * 16)
    monkeypatch.setattr(bench, "ROOT", str(root))
    sha = bench.kernel_source_hash()
    assert bench.read_traffic("w", 1_000_000) is None                 # taken on other sources
    (root / "profiles" / "gemv_w.md").write_text(f"- kernel_source_sha: {sha}\n- dram_over_algorithmic: 1.0015\n")
    assert bench.read_traffic("w", 1_000_000) == 1_001_500
    # only the GEMV kernels' own sources count towards the hash
    (root / "gemm_uq_gb300" / "csrc" / "uq_tc.cu").write_text("changed\n")
    assert bench.kernel_source_hash() == sha
    (root / "gemm_uq_gb300" / "csrc" / "uq_gemv.cuh").write_text("kernel a, changed\n")
    assert bench.kernel_source_hash() != sha and bench.read_traffic("w", 1_000_000) is None
    assert bench.read_traffic("missing", 1_000_000) is None
    assert bench.read_share("w") == 0.912 and bench.read_share("missing") is None


def test_dominant_kernel_follows_the_library_routing():
    step = [(14336, 4096), (4096, 14336)]
    assert bench.dominant_kernel("INT4_ASYM", 128, 1, step) == "gemv_warp_kernel<INT4_ASYM,GB=8>"
    assert bench.dominant_kernel("INT4_SYM", 32, 1, step) == "gemv_warp_kernel<INT4_SYM,GB=2>"
    assert bench.dominant_kernel("INT4_ASYM", 128, 8, step) == "gemv_mma_kernel<INT4_ASYM,GB=8>"
    assert bench.dominant_kernel("INT8_SYM", 128, 1, step) == "gemv_mma_kernel<INT8_SYM,GB=8>"
    assert bench.dominant_kernel("K4", 256, 1, step) == "gemv_mma_kernel<K4,GB=2>"
    assert bench.dominant_kernel("INT4_ASYM", 128, 12, step) == "gemm_mma_kernel<INT4_ASYM,16 columns>"
    assert bench.dominant_kernel("K4", 256, 32, step) == "gemm_mma_kernel<K4,32 columns>"
    assert bench.dominant_kernel("INT4_ASYM", 128, 64, step) == "tc_kernel<INT4_ASYM,64>"
    assert bench.dominant_kernel("NF4", 64, 16, [(8192, 8192)]) == "tc_kernel<NF4,16>"
    # a K that is not a multiple of the code tile keeps 16+ rows on the GEMV
    assert bench.dominant_kernel("NF4", 64, 20, [(4096, 4096 + 64)]) == "gemv_mma_kernel<NF4,GB=4>"


def test_roofline_time_is_the_slower_bound():
    assert bench.roofline_time_s(6786.6e9, 0, 6786.6, 1915.3) == 1.0
    assert bench.roofline_time_s(0, 1915.3e12, 6786.6, 1915.3) == 1.0
    assert bench.roofline_time_s(6786.6e9, 3830.6e12, 6786.6, 1915.3) == 2.0
