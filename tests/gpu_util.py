"""Helpers for the GPU parity tests: tolerances, guard bands, device copies."""
import numpy as np
import pytest
import torch

# Layer-level bound for bf16 inputs with fp32 accumulation.
LAYER_RTOL = 2e-2
# Standalone fp32-output kernels (products of bf16 values are exact in fp32; only
# the order of fp32 additions differs from the fp64 oracle).
KERNEL_RTOL = 1e-3
# bf16-rounded outputs: round-to-nearest-even costs at most 2^-9 relative.
BF16_REL = 2.0 ** -7

GUARD = 1024  # elements of sentinel on each side of a guarded output buffer


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import expert_adapter_gemms_gb300 as m
    m.lib()
    return m


def dev(t):
    return None if t is None else t.to("cuda").contiguous()


def f64(t):
    return t.detach().to("cpu").to(torch.float64).numpy()


def assert_close(gpu, ref, rtol, what=""):
    g = f64(gpu) if isinstance(gpu, torch.Tensor) else np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    err = np.abs(g - r)
    bound = rtol * (1.0 + np.abs(r))
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance; worst at {i}: "
                             f"gpu={g[i]!r} ref={r[i]!r} err={err[i]:.3g} bound={bound[i]:.3g}")
    return float((err / (1.0 + np.abs(r))).max()) if err.size else 0.0


def assert_bf16_close(gpu, ref, what="", atol=1e-4):
    g = f64(gpu)
    r = np.asarray(ref, dtype=np.float64)
    err = np.abs(g - r)
    bound = BF16_REL * np.abs(r) + atol
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} bf16 elements out of tolerance; worst at "
                             f"{i}: gpu={g[i]!r} ref={r[i]!r}")


class Guarded:
    """A device buffer with sentinel bands on both sides, checked after use."""

    def __init__(self, shape, dtype, fill=0.0):
        n = int(np.prod(shape))
        self.raw = torch.empty(n + 2 * GUARD, dtype=dtype, device="cuda")
        if dtype.is_floating_point:
            self.sent = torch.tensor(-12345.5, dtype=dtype)
        else:
            self.sent = torch.tensor(-123456789, dtype=dtype)
        self.raw[:GUARD] = self.sent
        self.raw[GUARD + n:] = self.sent
        self.t = self.raw[GUARD:GUARD + n].view(*shape)
        self.t.fill_(fill)

    def check(self):
        torch.cuda.synchronize()
        lo = self.raw[:GUARD].cpu()
        hi = self.raw[-GUARD:].cpu()
        assert bool((lo == self.sent).all()) and bool((hi == self.sent).all()), \
            "write outside the output buffer"
