"""Seeded synthetic inputs for the FP4 block-scaled quantize-and-multiply path.

Both the CUDA path and the CPU oracle take their inputs from here.  This module
holds no arithmetic of the method: it only draws tensors with the shapes and
value distributions of the workloads the pages describe, in binary32 from a
seeded ``torch.Generator`` and then rounded once to BF16 (nearest-even).

Workloads (sizes are parameters so that parity tests can draw small cases
with the same distributions):

* ``tiny``            X ~ N(0,1) with 0.1% of entries x50, W ~ N(0, 0.02).
* ``forward_layer``   X ~ N(0,1) with 1% of channels scaled by LogNormal(0,1),
                      W ~ N(0, 0.02).
* ``backward_sr``     dY ~ Student-t(3) * 1e-4, X as ``tiny``, W as above.
* ``down_proj_8b``    X = |N(0,1)| * N(0,1) (post-SwiGLU), W ~ N(0, 0.014),
                      dY ~ Student-t(3) * 1e-4.
* ``sweep_operand``   N(0,1) with 1% of entries x50.

Draw order within a workload is fixed as listed; outlier positions come from
``randperm`` on the same generator.  ``sweep_operand`` can also draw on a CUDA
device (its own seeded generator there): the same distribution, other values,
for timing runs whose operands are too large to draw on the host quickly.
"""
import torch


def _gen(seed, device="cpu"):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal(shape, std, g):
    return torch.randn(shape, generator=g, dtype=torch.float32, device=g.device) * std


def _scale_entries(x, frac, factor, g):
    n = int(round(frac * x.numel()))
    if n:
        idx = torch.randperm(x.numel(), generator=g, device=g.device)[:n]
        x.view(-1)[idx] *= factor
    return x


def _scale_channels_lognormal(x, frac, g):
    """Multiply round(frac * cols) randomly chosen columns by exp(N(0,1))."""
    cols = x.shape[1]
    n = int(round(frac * cols))
    if n:
        idx = torch.randperm(cols, generator=g)[:n]
        x[:, idx] *= torch.exp(torch.randn(n, generator=g))
    return x


def _student_t(shape, nu, g):
    """Student-t with nu degrees of freedom: Z / sqrt(V / nu), V ~ chi^2(nu)."""
    z = torch.randn(shape, generator=g)
    v = torch.zeros(shape)
    for _ in range(nu):
        v += torch.randn(shape, generator=g) ** 2
    return z / torch.sqrt(v / nu)


def bf16(x):
    return x.to(torch.bfloat16)


def tiny(seed=0, M=256, K=256, N=256):
    g = _gen(seed)
    x = _scale_entries(_normal((M, K), 1.0, g), 0.001, 50.0, g)
    w = _normal((N, K), 0.02, g)
    return dict(X=bf16(x), W=bf16(w))


def forward_layer(seed=0, M=8192, K=4096, N=4096):
    g = _gen(seed)
    x = _scale_channels_lognormal(_normal((M, K), 1.0, g), 0.01, g)
    w = _normal((N, K), 0.02, g)
    return dict(X=bf16(x), W=bf16(w))


def backward_sr(seed=0, M=8192, K=4096, N=4096):
    g = _gen(seed)
    dy = _student_t((M, N), 3, g) * 1e-4
    x = _scale_entries(_normal((M, K), 1.0, g), 0.001, 50.0, g)
    w = _normal((N, K), 0.02, g)
    return dict(dY=bf16(dy), X=bf16(x), W=bf16(w))


def down_proj_8b(seed=0, M=8192, K=14336, N=4096):
    g = _gen(seed)
    x = torch.abs(_normal((M, K), 1.0, g)) * _normal((M, K), 1.0, g)
    w = _normal((N, K), 0.014, g)
    dy = _student_t((M, N), 3, g) * 1e-4
    return dict(X=bf16(x), W=bf16(w), dY=bf16(dy))


def sweep_operand(rows, cols, seed=7, device="cpu"):
    g = _gen(seed, device)
    return bf16(_scale_entries(_normal((rows, cols), 1.0, g), 0.01, 50.0, g))


def mxfp4_copy(rows, cols, seed=11, spread=20):
    """Random bytes in the shape of an MXFP4-b32 row-wise copy, for the FP8
    re-encoding: payload [rows][cols/2] (uniform bytes, so every E2M1 code
    and sign appears) and E8M0 codes [rows][cols/32].  Per 128 columns the
    four codes are a base in [spread, 254] minus 0..spread each, so the
    blocks of one FP8 block lie up to `spread` binades apart; a few codes are
    pinned to the extremes 0, 254 and 255.  Returns uint8 tensors."""
    g = _gen(seed)
    q = torch.randint(0, 256, (rows, cols // 2), generator=g, dtype=torch.int32)
    nb = cols // 128
    base = torch.randint(spread, 255, (rows, nb, 1), generator=g, dtype=torch.int32)
    off = torch.randint(0, spread + 1, (rows, nb, 4), generator=g, dtype=torch.int32)
    sf = (base - off).reshape(rows, cols // 32)
    if sf.numel() >= 12:
        flat = sf.view(-1)
        idx = torch.randperm(flat.numel(), generator=g)[:3]
        flat[idx] = torch.tensor([0, 254, 255], dtype=torch.int32)
    return q.to(torch.uint8), sf.to(torch.uint8)


def fp4_copy(rows, cols, block, max_code, seed=13):
    """Random bytes in the shape of a row-wise FP4 copy with plain-layout
    scales: payload [rows][cols/2] (uniform bytes: every E2M1 code and sign)
    and scale codes [rows][cols/block] uniform in 0 .. max_code.  Returns
    uint8 tensors."""
    g = _gen(seed)
    q = torch.randint(0, 256, (rows, cols // 2), generator=g, dtype=torch.int32)
    sf = torch.randint(0, max_code + 1, (rows, cols // block), generator=g, dtype=torch.int32)
    return q.to(torch.uint8), sf.to(torch.uint8)
