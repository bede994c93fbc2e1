"""ctypes front end of the seeded generator (gen/synth.c).

Everything returned is a numpy array in the canonical layouts that both the
oracle and the CUDA path take as input:

* Q4 matrix: uint8 [rows, k/256*144] (super-blocks along k, row-major).
* fp32 vectors / matrices: float32 with the tensor's shape.
* KV pool: per attention layer, per page, per kv head, per page slot, dh values;
  fp16 as uint16 bit patterns, or int8 codes + binary16 scales per 32 values.
* Gated-DeltaNet state per sequence: float32 [n_gdn][hv][dv][dk] and the
  convolution history float32 [n_gdn][conv_w-1][conv_ch].
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from .configs import FA, GDN, PAGE_TOKENS, model_dims, tensor_inventory

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_SO = os.path.join(_HERE, "libsynth.so")

_CFLAGS = ["-O2", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off", "-pthread"]


def build(force: bool = False) -> str:
    """Compile the generator library in-tree (gcc, a second or two)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        u64, i64, i32, dbl, vp = (ctypes.c_uint64, ctypes.c_int64, ctypes.c_int,
                                  ctypes.c_double, ctypes.c_void_p)
        L.synth_q4.argtypes = [u64, u64, i64, i64, dbl, vp, i32]
        L.synth_normal_f64.argtypes = [u64, u64, i64, dbl, vp]
        L.synth_normal_f32.argtypes = [u64, u64, i64, dbl, dbl, vp, i32]
        L.synth_normal_f16.argtypes = [u64, u64, i64, dbl, dbl, vp, i32]
        L.synth_q8_blocks.argtypes = [u64, u64, i64, vp, vp, i32]
        L.synth_uniform_int.argtypes = [u64, u64, i64, ctypes.c_uint32, vp]
        L.synth_permutation.argtypes = [u64, u64, i64, vp]
        L.synth_raw.argtypes = [u64, u64, i64, vp]
        for f in ("synth_q4", "synth_normal_f64", "synth_normal_f32", "synth_normal_f16",
                  "synth_q8_blocks", "synth_uniform_int", "synth_permutation", "synth_raw"):
            getattr(L, f).restype = ctypes.c_int
        _lib = L
    return _lib


def _threads(n=None):
    return int(n or os.environ.get("SYNTH_THREADS", os.cpu_count() or 1))


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def q4_nbytes(rows: int, k: int) -> int:
    return rows * (k // 256) * 144


def q4_matrix(seed, tid, rows, k, sigma, nthreads=None) -> np.ndarray:
    out = np.empty((rows, (k // 256) * 144), dtype=np.uint8)
    rc = lib().synth_q4(seed, tid, rows, k, sigma, _ptr(out), _threads(nthreads))
    if rc:
        raise ValueError("q4 matrix needs k % 256 == 0")
    return out


def normal_f64(seed, tid, n, sigma=1.0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    lib().synth_normal_f64(seed, tid, n, sigma, _ptr(out))
    return out


def normal_f32(seed, tid, shape, mean=0.0, sigma=1.0, nthreads=None) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    lib().synth_normal_f32(seed, tid, out.size, mean, sigma, _ptr(out), _threads(nthreads))
    return out


def normal_f16_bits(seed, tid, shape, mean=0.0, sigma=1.0, nthreads=None) -> np.ndarray:
    out = np.empty(shape, dtype=np.uint16)
    lib().synth_normal_f16(seed, tid, out.size, mean, sigma, _ptr(out), _threads(nthreads))
    return out


def q8_blocks(seed, tid, codes_shape, nthreads=None):
    codes = np.empty(codes_shape, dtype=np.int8)
    assert codes.size % 32 == 0
    scales = np.empty(codes_shape[:-1] + (codes_shape[-1] // 32,), dtype=np.uint16)
    lib().synth_q8_blocks(seed, tid, codes.size // 32, _ptr(codes), _ptr(scales),
                          _threads(nthreads))
    return codes, scales


def uniform_tokens(seed, tid, count, vocab) -> np.ndarray:
    out = np.empty(count, dtype=np.int32)
    lib().synth_uniform_int(seed, tid, count, vocab, _ptr(out))
    return out


def permutation(seed, tid, n) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    lib().synth_permutation(seed, tid, n, _ptr(out))
    return out


def raw_draws(seed, tid, n) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    lib().synth_raw(seed, tid, n, _ptr(out))
    return out


def make_weights(m: dict, seed: int = 0, norm_jitter: float = 0.0, nthreads=None,
                 only=None) -> dict:
    """All canonical tensors of model m.

    Q4 matrices ~ N(0, weight_sigma) quantised; convolution taps ~ N(0, 0.5);
    norm gains = 1 (or 1 + N(0, norm_jitter) when a test wants them to matter).
    """
    out = {}
    for name, tid, kind, shape in tensor_inventory(m):
        if only is not None and name not in only:
            continue
        if kind == "q4":
            out[name] = q4_matrix(seed, tid, shape[0], shape[1], m["weight_sigma"], nthreads)
        elif name.endswith("conv_w"):
            out[name] = normal_f32(seed, tid, shape, 0.0, 0.5, nthreads)
        else:  # norm gains
            if norm_jitter:
                out[name] = normal_f32(seed, tid, shape, 1.0, norm_jitter, nthreads)
            else:
                out[name] = np.ones(shape, dtype=np.float32)
    return out


def make_pool(m: dict, n_pages: int, kv_q8: int) -> dict:
    """Zero KV pool arrays: one attention layer per full-attention layer, plus
    one for the multi-token-prediction block when the model has it."""
    d = model_dims(m)
    nl = d["n_fa"] + (1 if m.get("has_mtp") else 0)
    shape = (nl, n_pages, m["hkv"], PAGE_TOKENS, m["dh"])
    if kv_q8:
        sshape = shape[:-1] + (m["dh"] // 32,)
        return dict(kq=np.zeros(shape, np.int8), vq=np.zeros(shape, np.int8),
                    ks=np.zeros(sshape, np.uint16), vs=np.zeros(sshape, np.uint16))
    return dict(k=np.zeros(shape, np.uint16), v=np.zeros(shape, np.uint16))


def fill_pool(pool: dict, seed: int, nthreads=None) -> None:
    """Synthetic cache contents for every page: K, V ~ N(0,1) (stored post-RoPE),
    as binary16, or as q8 blocks (codes ~ N(0,1)*127/A, scale f16(A/127))."""
    if "k" in pool:
        pool["k"][...] = normal_f16_bits(seed, 50001, pool["k"].shape, nthreads=nthreads)
        pool["v"][...] = normal_f16_bits(seed, 50002, pool["v"].shape, nthreads=nthreads)
    else:
        c, s = q8_blocks(seed, 50003, pool["kq"].shape, nthreads)
        pool["kq"][...] = c
        pool["ks"][...] = s
        c, s = q8_blocks(seed, 50004, pool["vq"].shape, nthreads)
        pool["vq"][...] = c
        pool["vs"][...] = s


def make_seq_states(m: dict, seed: int, seq: int, nthreads=None):
    """Recurrent state of one sequence: S ~ N(0,1), convolution history ~ N(0,1)."""
    d = model_dims(m)
    S = normal_f32(seed, 60000 + seq, (d["n_gdn"], m["hv"], m["dv"], m["dk"]), nthreads=nthreads)
    conv = normal_f32(seed, 61000 + seq, (d["n_gdn"], m["conv_w"] - 1, d["conv_ch"]),
                      nthreads=nthreads)
    return S, conv


def seq_pages(n_cached: int, page_ids) -> np.ndarray:
    n = (n_cached + PAGE_TOKENS - 1) // PAGE_TOKENS
    return np.asarray(page_ids[:n], dtype=np.int32)


__all__ = ["FA", "GDN"]
