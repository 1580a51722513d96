"""Child process of tests/test_zz_no_alloc.py (run with the library path as argv[1]).

A caller that cannot allocate device memory calls moe_lora_layer_noalloc; such a
caller may also tear its CUDA context down and start again (cudaDeviceReset) during
the life of the process. The library-held array then sits at a new device address in
the new context, and the entry point must look it up again. This script checks that
in a fresh process, without torch (whose device state would not survive the reset):
inputs are drawn with numpy, copied with the CUDA runtime, and each
moe_lora_layer_noalloc result is compared bit for bit with moe_lora_layer (the same
kernels on a caller workspace), once before and once after a cudaDeviceReset.
Prints "ok" on success; any mismatch or CUDA error exits non-zero.
"""
import ctypes
import sys

import numpy as np

P, I, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
H2D, D2H = 1, 2


def bf16_bits(a):
    """fp32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def main(lib_path):
    lib = ctypes.CDLL(lib_path)
    rt = ctypes.CDLL("libcudart.so.13")  # the runtime the library itself loaded
    rt.cudaMalloc.argtypes = [ctypes.POINTER(P), SZ]
    rt.cudaMemcpy.argtypes = [P, P, SZ, I]
    rt.cudaFree.argtypes = [P]
    for fn in (rt.cudaMalloc, rt.cudaMemcpy, rt.cudaFree, rt.cudaDeviceSynchronize,
               rt.cudaDeviceReset):
        fn.restype = I
    noalloc = lib.moe_lora_layer_noalloc
    noalloc.restype = I
    noalloc.argtypes = [P, P, P, P, P, I, I, I, I, I, P, P, P, P, P, P, I, I, P, I, P, P]
    layer = lib.moe_lora_layer
    layer.restype = I
    layer.argtypes = [P, P, P, P, P, I, I, I, I, I, P, P, P, P, P, P, I, I, P, I, P, SZ, P]
    wsize = lib.moe_lora_workspace_size
    wsize.restype = SZ
    wsize.argtypes = [I] * 7

    def ok(rc, what):
        if rc != 0:
            raise SystemExit(f"{what} failed with {rc}")

    T, H, Ih, E, k, L, r = 16, 128, 64, 4, 2, 2, 16

    def one_round(seed):
        rng = np.random.default_rng(seed)
        host = {
            "x": bf16_bits(rng.standard_normal((T, H))),
            "logits": rng.standard_normal((T, E)).astype(np.float32),
            "ta": np.array([l % (L + 1) - 1 for l in range(T)], dtype=np.int32),
            "W1": bf16_bits(rng.standard_normal((E, 2 * Ih, H)) * 0.05),
            "W2": bf16_bits(rng.standard_normal((E, H, Ih)) * 0.05),
            "A1": bf16_bits(rng.standard_normal((L, E, r, H)) * 0.1),
            "B1": bf16_bits(rng.standard_normal((L, E, 2 * Ih, r)) * 0.1),
            "A2": bf16_bits(rng.standard_normal((L, E, r, Ih)) * 0.1),
            "B2": bf16_bits(rng.standard_normal((L, E, H, r)) * 0.1),
        }
        dev = {}
        for name, a in host.items():
            p = P()
            ok(rt.cudaMalloc(ctypes.byref(p), a.nbytes), "cudaMalloc")
            ok(rt.cudaMemcpy(p, a.ctypes.data, a.nbytes, H2D), "cudaMemcpy")
            dev[name] = p
        nws = wsize(T, k, E, L, H, Ih, r)
        for name, n in (("y0", T * H * 4), ("y1", T * H * 4), ("ws", nws), ("err", 4)):
            p = P()
            ok(rt.cudaMalloc(ctypes.byref(p), n), "cudaMalloc")
            dev[name] = p
        zero = np.zeros(256, dtype=np.uint8)
        ok(rt.cudaMemcpy(dev["ws"], zero.ctypes.data, 256, H2D), "cudaMemcpy")  # error word
        d = dev
        ok(layer(d["x"], d["logits"], None, None, d["ta"], T, H, Ih, E, k, d["W1"], d["W2"],
                 d["A1"], d["B1"], d["A2"], d["B2"], L, r, d["y0"], 1, d["ws"], nws, None),
           "moe_lora_layer")
        ok(noalloc(d["x"], d["logits"], None, None, d["ta"], T, H, Ih, E, k, d["W1"], d["W2"],
                   d["A1"], d["B1"], d["A2"], d["B2"], L, r, d["y1"], 1, d["err"], None),
           "moe_lora_layer_noalloc")
        ok(rt.cudaDeviceSynchronize(), "cudaDeviceSynchronize")
        y0 = np.empty((T, H), dtype=np.float32)
        y1 = np.empty((T, H), dtype=np.float32)
        err = np.zeros(1, dtype=np.uint32)
        ok(rt.cudaMemcpy(y0.ctypes.data, d["y0"], y0.nbytes, D2H), "cudaMemcpy")
        ok(rt.cudaMemcpy(y1.ctypes.data, d["y1"], y1.nbytes, D2H), "cudaMemcpy")
        ok(rt.cudaMemcpy(err.ctypes.data, d["err"], 4, D2H), "cudaMemcpy")
        if int(err[0]) != 0:
            raise SystemExit(f"device error word {int(err[0]):#x}")
        if not np.isfinite(y0).all() or not np.array_equal(y0.view(np.uint32), y1.view(np.uint32)):
            raise SystemExit("moe_lora_layer_noalloc differs from moe_lora_layer")
        for p in dev.values():
            ok(rt.cudaFree(p), "cudaFree")

    one_round(1)
    ok(rt.cudaDeviceReset(), "cudaDeviceReset")
    one_round(2)
    print("ok")


if __name__ == "__main__":
    main(sys.argv[1])
