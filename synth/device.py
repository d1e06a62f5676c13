"""ctypes binding of libkfsynth.so: fills device buffers with the synthetic streams."""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import recipes
from .build import LIB

_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError("libkfsynth.so is not built; run __graft_entry__.build()")
        _lib = ctypes.CDLL(LIB)
        f = _lib.kfsynth_fill
        f.restype = ctypes.c_int
        f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                      ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_uint64,
                      ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p]
    return _lib


def fill(out_ptr: int, dtype: str, rows: int, cols: int, ld: int, row0: int, total_cols: int,
         col0: int, seed: int, std_ptr: int, scale: float, stream: int) -> None:
    rc = lib().kfsynth_fill(ctypes.c_void_p(out_ptr), 0 if dtype == "bf16" else 1, rows, cols, ld,
                            row0, total_cols, col0, ctypes.c_uint64(seed & ((1 << 64) - 1)),
                            ctypes.c_void_p(std_ptr), float(scale), ctypes.c_void_p(stream))
    if rc != 0:
        raise RuntimeError("kfsynth_fill failed with cudaError %d" % rc)


def stream_on_device(wl: recipes.Workload, site: recipes.Site, t0: int, t1: int, torch, device="cuda"):
    """Rows t0..t1-1 of a calibration stream as a device tensor of the workload's dtype."""
    dt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    out = torch.empty((t1 - t0, site.d), dtype=dt, device=device)
    std = torch.from_numpy(recipes.site_std(wl, site)).to(device)
    fill(out.data_ptr(), wl.dtype, t1 - t0, site.d, site.d, t0, site.d, 0,
         recipes.stream_seed(wl, site), std.data_ptr(), 1.0, torch.cuda.current_stream().cuda_stream)
    return out


def weight_on_device(wl: recipes.Workload, unit: recipes.Unit, torch, device="cuda"):
    """The whole weight the unit belongs to (for an attention head: the full matrix)."""
    dt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    wm, wn = unit.weight_shape
    out = torch.empty((wm, wn), dtype=dt, device=device)
    fill(out.data_ptr(), wl.dtype, wm, wn, wn, 0, wn, 0,
         recipes.weight_seed(wl, unit), 0, float(recipes.weight_std(wl)),
         torch.cuda.current_stream().cuda_stream)
    return out


def weights_on_device(wl: recipes.Workload, torch, device="cuda"):
    """Every weight of a workload, keyed by weight name (heads share their matrix)."""
    out = {}
    for u in wl.units:
        if u.weight not in out:
            out[u.weight] = weight_on_device(wl, u, torch, device)
    return out


def rows_fn(wl: recipes.Workload, torch, device="cuda"):
    """A callable (site, t0, t1) -> device rows, generating calibration chunks on demand."""
    def rows(name, t0, t1):
        return stream_on_device(wl, wl.sites[name], t0, t1, torch, device)
    return rows
