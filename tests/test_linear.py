"""FP4Linear: sample-and-hold policy (CPU) and forward / backward against the
oracle on the GPU ("UE5M3 FP4 Block Scaling for Stable Language Model
Pretraining", Approach: held amax refreshed every D steps, SR on the upstream
gradient, 2D weight tiles)."""
import numpy as np
import pytest
import torch

import fp4_block_scaled_quantize_gb300 as fq
from fp4_block_scaled_quantize_gb300 import inputs
from fp4_block_scaled_quantize_gb300.linear import AmaxCache, FP4Linear
import oracle as orc
from gpu_util import ORC_FMT, f32, need_gpu

UE, NV, MX = fq.FP4_FMT_UE5M3_B16, fq.FP4_FMT_NVFP4_B16, fq.FP4_FMT_MXFP4_B32


def test_sample_and_hold_schedule():
    c = AmaxCache(50, "cpu")
    assert c.due(7)                      # nothing held yet: first step refreshes
    c.last_refresh = 7
    due = [s for s in range(8, 200) if c.due(s)]
    assert due == [50, 100, 150]
    c1 = AmaxCache(1, "cpu")             # D = 1 is current scaling
    c1.last_refresh = 0
    assert all(c1.due(s) for s in range(1, 20))
    with pytest.raises(ValueError):
        AmaxCache(0, "cpu")


def test_amax_cache_not_in_state_dict():
    m = FP4Linear(128, 64, device="cpu")
    assert set(m.state_dict().keys()) == {"weight"}
    assert m.p_w.block2d == 1 and m.p_x.block2d == 0
    assert m.p_dy.round_row == fq.FP4_ROUND_SR and m.p_dy.round_col == fq.FP4_ROUND_SR
    m2 = FP4Linear(128, 64, T_dy=2048.0, device="cpu", check_status=False)
    # the override reaches the Wgrad (transposed) copy of dY only
    assert m2.p_dy.T == 448.0 and m2.p_dy.T_col == 2048.0 and m2.p_x.T == 448.0
    assert m.p_dy.sr_seed != m2.p_dy.sr_seed     # distinct SR streams per module
    m2.next_step()
    assert m2.step == 1


def test_next_step_raises_on_a_recorded_device_condition(monkeypatch):
    import fp4_block_scaled_quantize_gb300.linear as L
    m = FP4Linear(128, 64, device="cpu")
    monkeypatch.setattr(L, "fp4_status_sync", lambda: fq.FP4_ERR_NONFINITE)
    with pytest.raises(fq.FP4Error):
        m.next_step()
    assert m.step == 0
    monkeypatch.setattr(L, "fp4_status_sync", lambda: fq.FP4_OK)
    m.next_step()
    assert m.step == 1


# ----------------------------------------------------------------- GPU parity

def _oracle_layer(X, W, dY, fmt, amax_x, amax_w, amax_dy, T_dy, offset, seed=42):
    of = ORC_FMT[fmt]
    x32, w32, dy32 = f32(X), f32(W), f32(dY)
    ox_r, ox_c = orc.quantize_transpose(x32, amax_x, amax_x, of)
    ow_r, ow_c = orc.quantize_transpose(w32, amax_w, amax_w, of, block2d=True)
    ody_r, ody_c = orc.quantize_transpose(dy32, amax_dy, amax_dy, of, T=448.0, T_col=T_dy,
                                          sr_row=True, sr_col=True, seed=seed, offset=offset)
    return (ox_r, ow_r), (ody_r, ow_c), (ody_c, ox_c)


def _check_bf16(y_gpu, oa, ob, fmt, K, name):
    """bf16 output of one GEMM against the oracle's probe-matched model
    rounded to bf16: within one bf16 ulp plus the GEMM tolerance."""
    Mo, No = y_gpu.shape
    mm, nn = np.meshgrid(np.arange(Mo), np.arange(No), indexing="ij")
    y_model, _, s_abs = orc.gemm_model(oa["q"], oa["sf"], ob["q"], ob["sf"], ORC_FMT[fmt], K,
                                       oa["s_dec"], ob["s_dec"], mm.ravel(), nn.ravel())
    g = y_gpu.detach().float().cpu().numpy().ravel().astype(np.float64)
    ym = torch.from_numpy(y_model).to(torch.bfloat16).float().numpy().astype(np.float64)
    tol = np.abs(ym) * 2.0 ** -8 + 1e-6 * s_abs
    err = np.abs(g - ym)
    assert np.all(err <= tol), f"{name}: max err {err.max()} ({np.sum(err > tol)} outside)"


@pytest.mark.gpu
@pytest.mark.parametrize("fmt", [UE, NV, MX])
def test_linear_forward_backward_matches_oracle(fmt):
    need_gpu()
    M, K, N = 256, 384, 192
    d = inputs.down_proj_8b(M=M, K=K, N=N)
    X, W, dY = d["X"], d["W"], d["dY"]
    T_dy = 2048.0 if fmt == UE else 448.0
    lin = FP4Linear(K, N, D=50, T_dy=T_dy, format=fmt)
    with torch.no_grad():
        lin.weight.copy_(W.cuda())
    x = X.cuda().requires_grad_(True)
    y = lin(x)
    y.backward(dY.cuda())
    assert fq.fp4_status_sync() == fq.FP4_OK
    assert y.dtype == torch.bfloat16 and x.grad.dtype == torch.bfloat16
    a32 = lambda t: float(np.max(np.abs(f32(t))))
    fp, dg, wg = _oracle_layer(X, W, dY, fmt, a32(X), a32(W), a32(dY), T_dy, offset=0,
                               seed=lin.p_dy.sr_seed)
    _check_bf16(y, *fp, fmt, K, "fprop")
    _check_bf16(x.grad, *dg, fmt, N, "dgrad")
    _check_bf16(lin.weight.grad, *wg, fmt, M, "wgrad")


@pytest.mark.gpu
def test_linear_holds_amax_between_refreshes():
    """Step 1 of a D = 50 schedule quantises with the amax taken at step 0,
    even though its input doubled; step 50 refreshes."""
    need_gpu()
    M, K, N = 128, 256, 128
    d = inputs.down_proj_8b(M=M, K=K, N=N)
    X0, W = d["X"], d["W"]
    X1 = (X0.float() * 2).to(torch.bfloat16)
    lin = FP4Linear(K, N, D=50, format=UE)
    with torch.no_grad():
        lin.weight.copy_(W.cuda())
        lin(X0.cuda())
        lin.next_step()
        y1 = lin(X1.cuda())
    a0 = float(np.max(np.abs(f32(X0))))
    aw = float(np.max(np.abs(f32(W))))
    assert lin.cache_x.last_refresh == 0
    assert float(lin.cache_x.row.item()) == a0
    fp, _, _ = _oracle_layer(X1, W, W, UE, a0, aw, aw, 448.0, 0)
    _check_bf16(y1, *fp, UE, K, "fprop with held amax")
    lin.step = 50
    with torch.no_grad():
        lin(X1.cuda())
    assert lin.cache_x.last_refresh == 50
    assert float(lin.cache_x.row.item()) == 2 * a0


def test_exact_fallback_policy_reads_the_status_word(monkeypatch):
    import fp4_block_scaled_quantize_gb300.linear as L
    with pytest.raises(ValueError):
        FP4Linear(128, 64, device="cpu", format=NV, exact_fallback=True)
    monkeypatch.setattr(L, "fp4_status_sync", lambda: fq.FP4_ERR_SCALE_WINDOW)
    assert L._window_missed("test") is True
    monkeypatch.setattr(L, "fp4_status_sync", lambda: fq.FP4_OK)
    assert L._window_missed("test") is False
    monkeypatch.setattr(L, "fp4_status_sync", lambda: fq.FP4_ERR_NONFINITE)
    with pytest.raises(fq.FP4Error):
        L._window_missed("test")
    p = fq.params(format=UE, T=2048.0, sf_layout=fq.FP4_SF_MMA, sr_seed=7, sr_offset=3,
                  round_row=fq.FP4_ROUND_SR)
    q = L._plain(p)
    assert q.sf_layout == fq.FP4_SF_PLAIN and p.sf_layout == fq.FP4_SF_MMA
    assert (q.format, q.T, q.sr_seed, q.sr_offset, q.round_row) == (UE, 2048.0, 7, 3,
                                                                    fq.FP4_ROUND_SR)


def _check_exact(y_gpu, oa, ob, fmt, K, name):
    """One GEMM of the exact path against the oracle's exact product: the
    binary32 accumulation bound (K/16 + 16) 2^-23 S plus the BF16 rounding of
    the output."""
    Mo, No = y_gpu.shape
    mm, nn = np.meshgrid(np.arange(Mo), np.arange(No), indexing="ij")
    _, ye, s_abs = orc.gemm_model(oa["q"], oa["sf"], ob["q"], ob["sf"], ORC_FMT[fmt], K,
                                  oa["s_dec"], ob["s_dec"], mm.ravel(), nn.ravel())
    g = y_gpu.detach().float().cpu().numpy().ravel().astype(np.float64)
    tol = (K / 16 + 16) * 2.0 ** -23 * s_abs + np.abs(ye) * 2.0 ** -8
    err = np.abs(g - ye)
    assert np.all(err <= tol), f"{name}: max err/tol {np.max(err / np.maximum(tol, 1e-300))}"


@pytest.mark.gpu
@pytest.mark.parametrize("wide", ["x", "dy"])
def test_linear_exact_fallback_outside_the_scale_window(wide):
    """A row of X (or of dY) with blocks ~22 binades apart misses the E4M3
    window: without the policy the step reports FP4_ERR_SCALE_WINDOW; with it
    the GEMMs that meet the miss run on the exact path and match the oracle's
    exact products of the same copies."""
    need_gpu()
    M, K, N = 256, 384, 192
    d = inputs.down_proj_8b(M=M, K=K, N=N)
    X, W, dY = f32(d["X"]), d["W"], f32(d["dY"])
    if wide == "x":
        X[0, 0:16] = 4096.0
        X[0, 16:32] *= 2.0 ** -12
    else:
        dY[0, 0:16] = 0.4
        dY[0, 16:32] *= 2.0 ** -12
    X, dY = torch.from_numpy(X).to(torch.bfloat16), torch.from_numpy(dY).to(torch.bfloat16)
    T_dy = 2048.0
    plain = FP4Linear(K, N, D=50, T_dy=T_dy, format=UE)
    lin = FP4Linear(K, N, D=50, T_dy=T_dy, format=UE, exact_fallback=True,
                    sr_seed=plain.p_dy.sr_seed)
    for m in (plain, lin):
        with torch.no_grad():
            m.weight.copy_(W.cuda())
    x0 = X.cuda().requires_grad_(True)
    plain(x0).backward(dY.cuda())
    with pytest.raises(fq.FP4Error) as e:
        plain.next_step()
    assert e.value.code == fq.FP4_ERR_SCALE_WINDOW
    x = X.cuda().requires_grad_(True)
    y = lin(x)
    y.backward(dY.cuda())
    lin.next_step()  # the miss was handled: nothing left in the status word
    a32 = lambda t: float(np.max(np.abs(f32(t))))
    fp, dg, wg = _oracle_layer(X, W, dY, UE, a32(X), a32(W), a32(dY), T_dy, offset=0,
                               seed=lin.p_dy.sr_seed)
    if wide == "x":
        _check_exact(y, *fp, UE, K, "fprop (exact path)")
    else:
        _check_bf16(y, *fp, UE, K, "fprop (tensor cores)")
    _check_exact(x.grad, *dg, UE, N, "dgrad (exact path)")
    _check_exact(lin.weight.grad, *wg, UE, M, "wgrad (exact path)")
