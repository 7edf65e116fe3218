"""FP4 linear layer: the recipe's forward and backward through the library.

"UE5M3 FP4 Block Scaling for Stable Language Model Pretraining", Approach and
Developer view:
  * one held-amax cache per operand (activation X, weight W, gradient dY),
    refreshed by sample-and-hold every D steps (D = 50 in the recipe, D = 1 is
    "current" scaling) and deliberately not serialised in checkpoints;
  * block scale target T (448 by default) with a per-module override for the
    upstream gradient's Wgrad copy (T = 2048 on the Wgrad-dY of the four
    final mixer.down_proj modules); the Dgrad copy of dY keeps T;
  * nearest-even everywhere except stochastic rounding on dY (both backward
    GEMMs), 2D 16x16 weight tiles so the forward and backward views agree;
  * fprop Y = X W^T, dgrad dX = dY W, wgrad dW = dY^T X on the FP4 tensor
    cores.

Every computation runs in libfp4gb300.so; this module only allocates
buffers, keeps the step counter and passes pointers.

Device-side conditions (a bounded wait that ran out, a non-finite amax, a
UE5M3 row outside the tensor core's scale window) are recorded in the
library's per-device status word, which stays set until it is read.
``FP4Linear.next_step()`` reads it once per step (outside the hot loop) and
raises ``FP4Error`` if anything was recorded; pass ``check_status=False`` to
leave that to the caller.

UE5M3 rows whose block scales span more binades than the tensor core's E4M3
scale path holds (the hardware has no UE5M3 scale type: "UE5M3 FP4 Block
Scaling ...", Limitations) raise the scale-window condition.  With
``exact_fallback=True`` the layer reads the status word after producing its
operands: on a miss, the forward or backward step produces plain-layout
copies (the same codes) and multiplies their exact BF16 dequantisations on
the BF16 tensor cores (``gemm_exact``).  Each forward and backward then costs
one host synchronisation; the BF16 input and weight are kept for the
backward pass.
"""
import itertools

import torch

from . import (FP4_ERR_SCALE_WINDOW, FP4_FMT_UE5M3_B16, FP4_FMT_UE5M3_B32, FP4_OK,
               FP4_ROUND_SR, FP4_SF_MMA, FP4_SF_PLAIN, FP4Error, _check, fp4_amax, fp4_status_sync,
               gemm, gemm_exact, params, quantize_transpose)

# Distinct stochastic-rounding streams per module: the default Philox key of
# the k-th FP4Linear built in this process is (42 << 32) | k, so two layers
# never draw the same random bits at the same element positions.
_module_index = itertools.count()


class AmaxCache:
    """Held amax of one operand: a device float32 pair (row view, transposed
    view), refreshed when ``step % D == 0``.  Kept out of ``state_dict`` on
    purpose: after a restart the first step is a refresh step."""

    def __init__(self, D, device, hadamard_n=0, hadamard_signs=0):
        if D < 1:
            raise ValueError("D must be >= 1")
        self.D = int(D)
        self.hadamard_n, self.hadamard_signs = hadamard_n, hadamard_signs
        self.row = torch.zeros(1, dtype=torch.float32, device=device)
        self.col = torch.zeros(1, dtype=torch.float32, device=device)
        self.last_refresh = None

    def due(self, step):
        return self.last_refresh is None or step % self.D == 0

    def update(self, x, step):
        """Refresh from x on refresh steps; hold otherwise.  Returns True if
        the cache was refreshed."""
        if not self.due(step):
            return False
        _check(fp4_amax(x, self.hadamard_n, self.hadamard_signs, self.row, self.col), "fp4_amax")
        self.last_refresh = step
        return True


def _plain(p):
    """The same producer options with plain-layout scales (UE5M3 codes kept,
    no remap): the exact path's operands."""
    q = type(p).from_buffer_copy(p)
    q.sf_layout = FP4_SF_PLAIN
    return q


def _window_missed(where):
    """Read (and clear) the status word: True on a UE5M3 scale-window miss;
    any other recorded condition raises."""
    st = fp4_status_sync()
    if st == FP4_ERR_SCALE_WINDOW:
        return True
    if st != FP4_OK:
        raise FP4Error(st, where)
    return False


class _FP4LinearFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, w, mod):
        x2 = x.reshape(-1, x.shape[-1]).contiguous()
        mod.cache_x.update(x2, mod.step)
        mod.cache_w.update(w, mod.step)
        xr, xc = quantize_transpose(x2, mod.cache_x.row, mod.cache_x.col, mod.p_x)
        wr, wc = quantize_transpose(w, mod.cache_w.row, mod.cache_w.col, mod.p_w)
        exact = mod.exact_fallback and _window_missed(f"FP4Linear step {mod.step} forward")
        if exact:
            xr, xc = quantize_transpose(x2, mod.cache_x.row, mod.cache_x.col, _plain(mod.p_x))
            wr, wc = quantize_transpose(w, mod.cache_w.row, mod.cache_w.col, _plain(mod.p_w))
            y = gemm_exact(xr, wr, out_dtype=torch.bfloat16)
        else:
            y = gemm(xr, wr, out_dtype=torch.bfloat16)
        ctx.x_shape = x.shape
        ctx.exact = exact
        keep = mod.exact_fallback and not exact  # the backward may still need plain copies
        ctx.saved = (xc, wc, mod, x2 if keep else None, w if keep else None)
        return y.reshape(*x.shape[:-1], w.shape[0])

    @staticmethod
    def backward(ctx, dy):
        xc, wc, mod, x2, w = ctx.saved
        dy2 = dy.reshape(-1, dy.shape[-1]).to(torch.bfloat16).contiguous()
        mod.cache_dy.update(dy2, mod.step)
        p = mod.p_dy
        p.sr_offset = mod.step & 0xFFFFFFFF  # fresh random bits every step
        dyr, dyc = quantize_transpose(dy2, mod.cache_dy.row, mod.cache_dy.col, p)
        exact = ctx.exact
        if mod.exact_fallback:
            exact = _window_missed(f"FP4Linear step {mod.step} backward") or exact
        if exact:
            # plain copies with the same codes (the SR counters do not depend
            # on the scale layout); X^T and W^T again if the forward pass ran
            # on the tensor-core path
            dyr, dyc = quantize_transpose(dy2, mod.cache_dy.row, mod.cache_dy.col, _plain(p))
            if not ctx.exact:
                xc = quantize_transpose(x2, mod.cache_x.row, mod.cache_x.col, _plain(mod.p_x))[1]
                wc = quantize_transpose(w, mod.cache_w.row, mod.cache_w.col, _plain(mod.p_w))[1]
            dx = gemm_exact(dyr, wc, out_dtype=torch.bfloat16)
            dw = gemm_exact(dyc, xc, out_dtype=torch.float32)
        else:
            dx = gemm(dyr, wc, out_dtype=torch.bfloat16)   # [M, K]
            dw = gemm(dyc, xc, out_dtype=torch.float32)    # [N, K]
        return dx.reshape(ctx.x_shape), dw.to(mod.weight.dtype), None


class FP4Linear(torch.nn.Module):
    """y = x W^T with the FP4 block-scaled recipe (no bias).

    in_features, out_features and the number of tokens per call must be
    multiples of 64 (the K dimension of every one of the three GEMMs).
    ``format`` is one of the library's FP4 formats (UE5M3 block 16 by
    default); ``T_dy`` is the per-module target for the upstream gradient's
    transposed (Wgrad) copy; ``sr_seed`` (default: distinct per module) keys
    the stochastic rounding of dY; ``exact_fallback`` (UE5M3 formats only)
    sends a step whose copies miss the E4M3 scale window through the exact
    dequantised path instead of reporting the miss.
    Call ``next_step()`` once per optimizer step to advance the
    sample-and-hold clock."""

    def __init__(self, in_features, out_features, D=50, T=448.0, T_dy=None,
                 format=FP4_FMT_UE5M3_B16, sr_seed=None, device="cuda", dtype=torch.bfloat16,
                 check_status=True, exact_fallback=False):
        super().__init__()
        if exact_fallback and format not in (FP4_FMT_UE5M3_B16, FP4_FMT_UE5M3_B32):
            raise ValueError("exact_fallback applies to the UE5M3 formats only")
        if sr_seed is None:
            sr_seed = (42 << 32) | next(_module_index)
        self.check_status = bool(check_status)
        self.exact_fallback = bool(exact_fallback)
        self.in_features, self.out_features = in_features, out_features
        self.weight = torch.nn.Parameter(
            torch.empty(out_features, in_features, device=device, dtype=dtype))
        torch.nn.init.normal_(self.weight, std=0.02)
        self.step = 0
        self.cache_x = AmaxCache(D, device)
        self.cache_w = AmaxCache(D, device)
        self.cache_dy = AmaxCache(D, device)
        self.p_x = params(format=format, T=T, sf_layout=FP4_SF_MMA)
        self.p_w = params(format=format, T=T, block2d=True, sf_layout=FP4_SF_MMA)
        # the override applies to the transposed (Wgrad) copy of dY only
        self.p_dy = params(format=format, T=T, T_col=T_dy if T_dy is not None else 0.0,
                           round_row=FP4_ROUND_SR, round_col=FP4_ROUND_SR, sr_seed=sr_seed,
                           sf_layout=FP4_SF_MMA)

    def next_step(self):
        """Advance the sample-and-hold clock; with check_status, first read
        (and clear) the device status word and raise FP4Error if a kernel
        recorded a condition since the last read.  Reading it waits for the
        current stream."""
        if self.check_status:
            st = fp4_status_sync()
            if st != FP4_OK:
                raise FP4Error(st, f"FP4Linear step {self.step}")
        self.step += 1

    def forward(self, x):
        if x.dtype != torch.bfloat16:
            x = x.to(torch.bfloat16)
        return _FP4LinearFn.apply(x, self.weight.to(torch.bfloat16).contiguous(), self)

    def extra_repr(self):
        return (f"in_features={self.in_features}, out_features={self.out_features}, "
                f"D={self.cache_x.D}")


__all__ = ["AmaxCache", "FP4Linear"]
