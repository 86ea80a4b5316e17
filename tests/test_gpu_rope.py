"""GPU parity of the fused RMSNorm + RoPE (uq_rmsnorm_rope, uq_rope_table) against the oracle.

Pass rule (oracle/rope.py): |y - y_ref| <= 2^-8 |y_ref| + 1e-4 (|n_i| + |n_partner|) + 1e-6, every
element.  Rows as hidden vectors (D = hidden size) and as single heads (D = head_dim), decode-sized and
bulk M, positions up to the table's end, and the table itself against float64 cos/sin.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

import gemm_uq_gb300 as uq  # noqa: E402
from oracle import rope as orope  # noqa: E402
from synth import activations, bf16_round  # noqa: E402
from tests.uq_helpers import device_x, y_to_f64  # noqa: E402

DEV = torch.device("cuda:0")


def _gamma(seed, D):
    g = np.random.default_rng([seed, 7]).normal(1.0, 0.1, D).astype(np.float32)
    return bf16_round(g)


@pytest.mark.parametrize("max_pos,head_dim,base", [(8192, 128, 10000.0), (1024, 64, 500000.0), (131072, 128, 500000.0)])
def test_rope_table_within_one_fp32_ulp(max_pos, head_dim, base):
    """Every entry within one fp32 ulp of the float64 cos / sin, plus the float64 angle's own rounding
    (a few units in 2^-53 of the angle: near a zero of cos or sin at a large angle that term dominates)."""
    t = uq.rope_table(max_pos, head_dim, base, device=DEV).cpu().numpy().astype(np.float64)
    p = np.arange(max_pos)
    a = orope.rope_angles(p, head_dim, base)
    want = np.stack([np.cos(a), np.sin(a)], axis=-1)
    ulp = np.spacing(np.abs(want).astype(np.float32)).astype(np.float64)
    cond = 8.0 * 2.0 ** -53 * np.maximum(a, 1.0)[..., None]
    assert np.all(np.abs(t - want) <= ulp + cond)


@pytest.mark.parametrize("M,D,head_dim", [(1, 4096, 128), (7, 4096, 128), (64, 1024, 64), (33, 8192, 128),
                                          (1024, 128, 128), (3, 16384, 256), (5, 48, 16)])
def test_rmsnorm_rope_parity(M, D, head_dim):
    max_pos, base, eps = 8192, 500000.0, 1e-5
    x = activations(900 + M, M, D)
    g = _gamma(901, D)
    pos = np.random.default_rng(902).integers(0, max_pos, M).astype(np.int32)
    pos[0] = max_pos - 1
    table = uq.rope_table(max_pos, head_dim, base, device=DEV)
    y = uq.rmsnorm_rope(device_x(x, DEV), device_x(g[None, :], DEV)[0].contiguous(), torch.from_numpy(pos).to(DEV),
                        table, head_dim, eps)
    y_ref, n = orope.rmsnorm_rope(x, g, pos, head_dim, eps, base)
    r = orope.error_ratio(y_to_f64(y), y_ref, n, head_dim)
    assert uq.device_fault() == 0
    assert np.isfinite(r).all() and r.max() <= 1.0, f"max error ratio {r.max():.3g}"


def test_rmsnorm_rope_in_place_and_deterministic():
    M, D, hd, max_pos, base, eps = 16, 4096, 128, 4096, 10000.0, 1e-6
    x = activations(910, M, D)
    g = _gamma(911, D)
    pos = np.arange(M, dtype=np.int32) * 37
    table = uq.rope_table(max_pos, hd, base, device=DEV)
    gd = device_x(g[None, :], DEV)[0].contiguous()
    pd = torch.from_numpy(pos).to(DEV)
    y = uq.rmsnorm_rope(device_x(x, DEV), gd, pd, table, hd, eps)
    xd = device_x(x, DEV)
    uq.rmsnorm_rope(xd, gd, pd, table, hd, eps, y=xd)                 # in place
    assert torch.equal(xd.view(torch.int16), y.view(torch.int16))
    y_ref, n = orope.rmsnorm_rope(x, g, pos, hd, eps, base)
    assert orope.error_ratio(y_to_f64(xd), y_ref, n, hd).max() <= 1.0


def test_rmsnorm_rope_position_outside_table_is_flagged():
    M, D, hd = 3, 256, 128
    x = device_x(activations(920, M, D), DEV)
    g = device_x(_gamma(921, D)[None, :], DEV)[0].contiguous()
    table = uq.rope_table(64, hd, 10000.0, device=DEV)
    pos = torch.tensor([0, 64, 5], dtype=torch.int32, device=DEV)    # 64 is one past the table
    y = torch.full((M, D), 3.0, dtype=torch.bfloat16, device=DEV)
    uq.rmsnorm_rope(x, g, pos, table, hd, 1e-5, y=y)
    assert uq.device_fault() == 8
    assert torch.all(y[1] == 3.0)                                     # that row is left as it was
    assert not torch.all(y[0] == 3.0) and not torch.all(y[2] == 3.0)


def test_rmsnorm_rope_rejects_bad_shapes():
    x = torch.zeros((2, 100), dtype=torch.bfloat16, device=DEV)
    table = uq.rope_table(8, 16, 10000.0, device=DEV)
    with pytest.raises(uq.UqError):
        uq.rmsnorm_rope(x, x[0].contiguous(), torch.zeros(2, dtype=torch.int32, device=DEV), table, 24, 1e-5)
