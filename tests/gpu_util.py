"""Helpers shared by the GPU parity tests (no method arithmetic here)."""
import numpy as np
import pytest
import torch

import fp4_block_scaled_quantize_gb300 as fq
import oracle as orc

# library format id -> oracle format id (each side keeps its own enum)
ORC_FMT = {fq.FP4_FMT_UE5M3_B16: orc.UE5M3, fq.FP4_FMT_NVFP4_B16: orc.NVFP4,
           fq.FP4_FMT_MXFP4_B32: orc.MXFP4, fq.FP4_FMT_UE5M3_B32: orc.UE5M3_B32}
UE_FORMATS = (fq.FP4_FMT_UE5M3_B16, fq.FP4_FMT_UE5M3_B32)


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def f32(x_bf16):
    """BF16 tensor -> float32 numpy (exact widening)."""
    return x_bf16.float().cpu().numpy()


def np_u8(t):
    return t.cpu().numpy().astype(np.uint8)


def mismatch_report(got, want, name):
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, (name, got.shape, want.shape)
    bad = np.argwhere(got != want)
    if len(bad):
        i = tuple(bad[0])
        raise AssertionError(f"{name}: {len(bad)} of {got.size} differ; first at {i}: "
                             f"gpu={got[i]} oracle={want[i]}")


def b16_view(fmt_lib, sf_plain):
    """Scales at block-16 granularity: the tensor-core layout stores the
    UE5M3 block-32 control's codes once per 16-element half."""
    return np.repeat(sf_plain, 2, 1) if fmt_lib == fq.FP4_FMT_UE5M3_B32 else sf_plain


def expect_sf(fmt_lib, sf_plain, q_plain, layout, remap):
    """Oracle-side expected scale bytes and shift for one copy."""
    if layout == fq.FP4_SF_PLAIN:
        return sf_plain.ravel(), None
    sf16 = b16_view(fmt_lib, sf_plain)
    if fmt_lib in UE_FORMATS and remap:
        e4, shift, fails = orc.remap_ue5m3(sf16, q_plain)
        return orc.sf_to_mma(e4), shift
    return orc.sf_to_mma(sf16), None


def remap_fails(fmt_lib, sf_plain, q_plain):
    """Blocks with no exact E4M3 image under the per-row shift (oracle)."""
    return orc.remap_ue5m3(b16_view(fmt_lib, sf_plain), q_plain)[2]


def set_device_scalar(v, device="cuda"):
    return torch.tensor([v], dtype=torch.float32, device=device)
