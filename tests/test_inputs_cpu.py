"""The seeded input recipe (the shapes and distributions every parity test and
the benchmark draw from) holds what it states: fixed seeds reproduce, the
distributions have their stated scale, outlier fraction and tails.  CPU only."""

import numpy as np
import torch

from fp4_block_scaled_quantize_gb300 import inputs


def _f(t):
    return t.float().numpy()


def test_seeds_reproduce_and_differ():
    a, b, c = inputs.tiny(seed=0), inputs.tiny(seed=0), inputs.tiny(seed=1)
    assert torch.equal(a["X"], b["X"]) and torch.equal(a["W"], b["W"])
    assert not torch.equal(a["X"], c["X"])
    assert a["X"].dtype == torch.bfloat16 and a["X"].shape == (256, 256)
    q1, s1 = inputs.mxfp4_copy(64, 512, seed=3)
    q2, s2 = inputs.mxfp4_copy(64, 512, seed=3)
    assert torch.equal(q1, q2) and torch.equal(s1, s2)


def test_tiny_and_sweep_outliers():
    # 0.1% (tiny) and 1% (sweep) of the entries multiplied by 50: N(0,1) alone
    # essentially never exceeds 6, an outlier does unless its draw was < 0.12
    x = _f(inputs.tiny(seed=0)["X"])
    n_out = round(0.001 * x.size)
    big = int((np.abs(x) > 6).sum())
    assert 0.75 * n_out <= big <= n_out
    s = _f(inputs.sweep_operand(512, 512, seed=7))
    n_out = round(0.01 * s.size)
    big = int((np.abs(s) > 6).sum())
    assert 0.75 * n_out <= big <= n_out
    core = s[np.abs(s) <= 6]
    assert abs(core.std() - 1.0) < 0.05 and abs(core.mean()) < 0.02


def test_down_proj_distributions():
    d = inputs.down_proj_8b(seed=0, M=512, K=1024, N=256)
    x, w, dy = _f(d["X"]), _f(d["W"]), _f(d["dY"])
    assert x.shape == (512, 1024) and w.shape == (256, 1024) and dy.shape == (512, 256)
    # X = |z1| z2: mean 0, second moment 1, symmetric
    assert abs(x.mean()) < 0.01 and abs((x * x).mean() - 1.0) < 0.03
    assert abs(w.std() - 0.014) < 0.0005
    # dY = t_3 * 1e-4: median |t_3| = 0.7649, and heavy tails (P(|t_3| > 10) ~ 0.2%)
    assert abs(np.median(np.abs(dy)) / 1e-4 - 0.7649) < 0.03
    tail = (np.abs(dy) > 10e-4).mean()
    assert 0.001 < tail < 0.004


def test_forward_layer_scales_one_percent_of_channels():
    d = inputs.forward_layer(seed=0, M=2048, K=1000, N=64)
    x = _f(d["X"])
    col_std = x.std(axis=0)
    off = np.abs(np.log(col_std)) > 0.15  # a column scaled by exp(N(0,1)) (|N| > 0.15 mostly)
    assert 5 <= int(off.sum()) <= 10       # round(0.01 * 1000) = 10 channels
    assert abs(np.median(col_std) - 1.0) < 0.02


def test_mxfp4_copy_structure():
    rows, cols, spread = 96, 1024, 12
    q, sf = inputs.mxfp4_copy(rows, cols, seed=5, spread=spread)
    assert q.shape == (rows, cols // 2) and sf.shape == (rows, cols // 32)
    s = sf.numpy().astype(int)
    flat = s.reshape(-1)
    assert {0, 254, 255} <= set(flat.tolist())
    # apart from the three pinned codes, the four codes of an FP8 block lie
    # within `spread` binades of each other
    blocks = s.reshape(rows, cols // 128, 4)
    span = blocks.max(axis=2) - blocks.min(axis=2)
    assert (span > spread).sum() <= 3
    # payload bytes cover every E2M1 code in both nibbles
    qb = q.numpy()
    assert len(np.unique(qb & 15)) == 16 and len(np.unique(qb >> 4)) == 16


def test_fp4_copy_structure():
    q, sf = inputs.fp4_copy(64, 512, 16, 0xF7, seed=3)
    assert q.shape == (64, 256) and sf.shape == (64, 32)
    assert q.dtype == torch.uint8 and sf.dtype == torch.uint8
    s = sf.numpy()
    assert s.max() == 0xF7 and s.min() == 0  # the whole code range, nothing above
    qb = q.numpy()
    assert len(np.unique(qb & 15)) == 16 and len(np.unique(qb >> 4)) == 16
    q2, sf2 = inputs.fp4_copy(64, 512, 16, 0xF7, seed=3)
    assert torch.equal(q, q2) and torch.equal(sf, sf2)
