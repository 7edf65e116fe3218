"""The GEMM sweep's every shape on the GPU path end to end: (M, N, K) in
{2048, 4096, 8192, 16384}^3 plus (8192, 14336, 4096) and (14336, 8192, 4096),
operands N(0,1) with 1% of entries x50 (drawn on the device with the sweep's
seeded generator), GPU amax -> GPU UE5M3-b16 producer -> GPU GEMM, checked on
sampled outputs against the probe-matched model of the oracle's copies of the
sampled rows (quantised under the oracle's amax of the whole operand):
|y - model| <= 1e-6 S, |y - exact| <= 1e-3 S."""
import numpy as np
import pytest
import torch

import fp4_block_scaled_quantize_gb300 as fq
from fp4_block_scaled_quantize_gb300 import inputs
import oracle as orc
from gpu_util import need_gpu

pytestmark = pytest.mark.gpu

SIZES = (2048, 4096, 8192, 16384)
SHAPES = [(m, n, k) for m in SIZES for n in SIZES for k in SIZES]
SHAPES += [(8192, 14336, 4096), (14336, 8192, 4096)]
_ops = {}


def _operand(role, rows, K):
    """GPU copy and the oracle's tensor scale of one sweep operand (cached)."""
    key = (role, rows, K)
    if key not in _ops:
        x = inputs.sweep_operand(rows, K, seed=7 if role == "A" else 8, device="cuda")
        a, _ = fq.amax(x)
        q = fq.quantize(x, a, fq.params(format=fq.FP4_FMT_UE5M3_B16, sf_layout=fq.FP4_SF_MMA))
        s_enc, s_dec = orc.tensor_scale(orc.UE5M3, 448.0, orc.amax(x.float().cpu().numpy()))
        assert q.s_dec.item() == np.float32(s_dec)
        _ops[key] = (x, q, s_enc, s_dec)
    return _ops[key]


def _oracle_rows(x, rows, s_enc, s_dec):
    """The oracle's row-wise copy of the given rows (a row's copy depends only
    on the row and the tensor scale)."""
    xr = x[torch.as_tensor(rows, device=x.device)].float().cpu().numpy()
    q, sf = orc.quantize_rows(xr, orc.UE5M3, s_enc, s_dec)
    return q, sf


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_sweep_shape_end_to_end(M, N, K):
    need_gpu()
    xa, qa, sea, sda = _operand("A", M, K)
    xb, qb, seb, sdb = _operand("B", N, K)
    y = fq.gemm(qa, qb)
    st = fq.fp4_status_sync()
    assert st == fq.FP4_OK, fq.STATUS_NAMES[st]
    rng = np.random.default_rng(M * 7 + N * 3 + K)
    mi = np.concatenate([rng.integers(0, M, 60), [0, M - 1, 0, M - 1]])
    ni = np.concatenate([rng.integers(0, N, 60), [0, N - 1, N - 1, 0]])
    ra, ia = np.unique(mi, return_inverse=True)
    rb, ib = np.unique(ni, return_inverse=True)
    q_a, sf_a = _oracle_rows(xa, ra, sea, sda)
    q_b, sf_b = _oracle_rows(xb, rb, seb, sdb)
    y_model, y_exact, s_abs = orc.gemm_model(q_a, sf_a, q_b, sf_b, orc.UE5M3, K, sda, sdb, ia, ib)
    g = y[torch.as_tensor(mi, device=y.device), torch.as_tensor(ni, device=y.device)]
    g = g.cpu().numpy().astype(np.float64)
    scale = np.maximum(s_abs, 1e-300)
    rel_model = np.abs(g - y_model.astype(np.float64)) / scale
    rel_exact = np.abs(g - y_exact) / scale
    assert rel_model.max() <= 1e-6, (M, N, K, rel_model.max())
    assert rel_exact.max() <= 1e-3, (M, N, K, rel_exact.max())
    if (M, N, K) == SHAPES[-1]:
        _ops.clear()
