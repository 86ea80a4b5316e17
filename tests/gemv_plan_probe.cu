// Host-only check of the small-M GEMV's work planner: compiles the planner's translation unit
// (linked with the stand-in launchers of gemv_plan_stubs.cu) and prints, per shape, the plan a
// GB300 (152 SMs) gets and the ring it leaves.  Runs on a machine without a GPU (no CUDA call is
// made).
#include "../gemm_uq_gb300/csrc/uq_gemv.cu"
#include <cstdio>
#include <cstdlib>

// argv: fmt M N K group a8 gated; prints "grid cta_rows launches warp ring_slots xmode pairs"
int main(int argc, char** argv) {
    if (argc != 8) return 2;
    const int fmt = atoi(argv[1]), M = atoi(argv[2]), N = atoi(argv[3]), K = atoi(argv[4]);
    const int group = atoi(argv[5]), a8 = atoi(argv[6]), gated = atoi(argv[7]);
    const uq::Layout L(N, K, fmt);
    uq::GemvArgs a = {};
    a.M = M; a.N = N; a.K = K; a.group = group; a.a8 = a8; a.gated = gated;
    a.NB = (gated ? 2 : 1) * L.NB; a.KB = L.KB; a.T = (long long)a.NB * L.KB;
    const int sms = 152;
    const int grid = uq::gemv_plan(a, fmt, sms);
    const bool warp = !a8 && uq::gemv_warp_route(fmt, M);
    int slots = 0, xmode = -1;
    if (!warp && grid > 0) {
        const int sxg = uq::gemv_mma_sx_groups(fmt, group, a.NB, a.KB, grid, a.cta_rows);
        xmode = uq::gemv_mma_xmode(fmt, K, group, M, sxg, a.cta_rows, a8 ? 1 : 2, !gated);
        slots = uq::gemv_mma_smem(fmt, K, group, M, sxg, a.cta_rows, xmode, a8 ? 1 : 2).S2;
    }
    printf("%d %d %d %d %d %d %d\n", grid, a.cta_rows, uq::gemv_launches(fmt, a), warp ? 1 : 0, slots, xmode,
           uq::gemv_mma_pairs(fmt, a8 != 0));
    return 0;
}
