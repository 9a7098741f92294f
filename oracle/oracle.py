"""Python face of the fp64 CPU oracle (oracle/vsa_oracle.c).

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only tests/, __graft_entry__.smoke()
and the CPU-baseline leg of bench.py may import this module.  It never imports
the product package and the product package never imports it.

The wrappers below only marshal numpy arrays into the C routines; every step of
the arithmetic is in vsa_oracle.c, which cites the passages it follows:

  lut_to_blockmask   VSA look-up table -> 0/1 block mask (set semantics)
  blockmask_to_lut   ascending compaction, pad -1
  masked_attention   token mask from block mask + variable_block_sizes, then
                     two-pass fp64 softmax attention; base-2 LSE; empty rows
                     give +0.0 and LSE_EMPTY
  vsa_forward        lut_to_blockmask followed by masked_attention
  jenga_forward      masked_attention on the shared bitmap
  masked_attention_bwd / vsa_backward
                     the fp64 gradients dq, dk, dv of the same forward for a given dout
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "vsa_oracle.c")
LIB = os.path.join(HERE, "libvsa_oracle.so")

# The finite sentinel written for rows with no attended key: -FLT_MAX, the
# most negative finite binary32, widened to double.
LSE_EMPTY = -float(np.finfo(np.float32).max)

_lib = None


def build(src: str = SRC, lib: str = LIB, openmp: bool = True) -> str:
    """Compile the oracle with the host C compiler (gcc, -O2, OpenMP when the
    toolchain has it).  No -march flags: the same source builds on x86_64 and
    aarch64 hosts and computes the same result."""
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-fno-fast-math"]
    tmp = lib + ".tmp%d" % os.getpid()
    cmd = base + (["-fopenmp"] if openmp else []) + [src, "-o", tmp, "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0 and openmp:
        cmd = base + [src, "-o", tmp, "-lm"]
        r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("oracle build failed:\n" + r.stderr)
    os.replace(tmp, lib)
    return lib


def _needs_build(lib: str, src: str) -> bool:
    return (not os.path.exists(lib)) or os.path.getmtime(lib) < os.path.getmtime(src)


def load(lib: str = LIB, src: str = SRC):
    """Load (building first if missing or stale) and declare the C symbols."""
    global _lib
    if lib == LIB and _lib is not None:
        return _lib
    if _needs_build(lib, src):
        build(src, lib)
    h = ctypes.CDLL(lib)
    P = ctypes.c_void_p
    i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
    h.oracle_num_threads.restype = i32
    h.oracle_num_threads.argtypes = []
    h.oracle_lut_to_blockmask.restype = None
    h.oracle_lut_to_blockmask.argtypes = [P, P, i64, i32, i32, P]
    h.oracle_blockmask_to_lut.restype = None
    h.oracle_blockmask_to_lut.argtypes = [P, i64, i32, i32, P, P]
    h.oracle_masked_attention.restype = None
    h.oracle_masked_attention.argtypes = [P, P, P, i32, i32, i32, i32, i32, i32, P, i64,
                                          i64, i32, P, f64, P, i64, P, P]
    h.oracle_masked_attention_bwd.restype = None
    h.oracle_masked_attention_bwd.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, i32, P,
                                              i64, i64, i32, P, f64, P, P, P]
    if lib == LIB:
        _lib = h
    return h


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads(h=None) -> int:
    return (h or load()).oracle_num_threads()


def lut_to_blockmask(q2k_idx, q2k_num, nb: int, h=None) -> np.ndarray:
    """q2k_idx [..., rows, max_kv], q2k_num [..., rows] -> int8 [..., rows, nb]."""
    h = h or load()
    idx = _c(q2k_idx, np.int32)
    num = _c(q2k_num, np.int32)
    max_kv = idx.shape[-1]
    rows = int(np.prod(num.shape))
    assert idx.size == rows * max_kv
    mask = np.empty(num.shape + (nb,), dtype=np.int8)
    h.oracle_lut_to_blockmask(_ptr(idx), _ptr(num), rows, max_kv, nb, _ptr(mask))
    return mask


def blockmask_to_lut(mask, max_kv: int, h=None):
    """int8 [..., rows, nb] -> (q2k_idx int32 [..., rows, max_kv], q2k_num int32 [..., rows])."""
    h = h or load()
    m = _c(mask, np.int8)
    nb = m.shape[-1]
    rows = int(np.prod(m.shape[:-1]))
    idx = np.empty(m.shape[:-1] + (max_kv,), dtype=np.int32)
    num = np.empty(m.shape[:-1], dtype=np.int32)
    h.oracle_blockmask_to_lut(_ptr(m), rows, nb, max_kv, _ptr(idx), _ptr(num))
    return idx, num


def all_qblocks(B: int, H: int, nb: int) -> np.ndarray:
    """Every (b, h, qb) triple, head-major."""
    b, hh, qb = np.meshgrid(np.arange(B), np.arange(H), np.arange(nb), indexing="ij")
    return np.stack([b.ravel(), hh.ravel(), qb.ravel()], axis=1).astype(np.int32)


def masked_attention(q_bits, k_bits, v_bits, blockmask, block: int, scale: float,
                     vbs=None, sel=None, h=None):
    """Oracle forward on bf16 bit patterns: q uint16 [B,Hq,Sq,D], k and v [B,Hkv,Sk,D]
    (Hq a multiple of Hkv; query head h reads key/value head h // (Hq // Hkv)).

    blockmask: int8 [B,Hq,nbq,nbk] (per head) or [nbq,nbk] (shared by all B,H),
    nbq = Sq // block, nbk = Sk // block.  vbs: int32 [nbk] or None (full blocks).
    sel: int32 [n,3] of (b,h,qb); default every q-block.
    Returns (out float64 [n,block,D], lse float64 [n,block]).
    """
    h = h or load()
    q = _c(q_bits, np.uint16)
    k = _c(k_bits, np.uint16)
    v = _c(v_bits, np.uint16)
    B, Hq, Sq, D = q.shape
    Bk, Hkv, Sk, Dk = k.shape
    assert v.shape == k.shape and Bk == B and Dk == D and Hq % Hkv == 0
    assert Sq % block == 0 and Sk % block == 0
    nbq, nbk = Sq // block, Sk // block
    m = _c(blockmask, np.int8)
    if m.ndim == 2:
        assert m.shape == (nbq, nbk)
        sb, sh = 0, 0
    else:
        assert m.shape == (B, Hq, nbq, nbk)
        sb, sh = Hq, 1
    vb = None if vbs is None else _c(vbs, np.int32)
    if vb is not None:
        assert vb.shape == (nbk,)
    s = all_qblocks(B, Hq, nbq) if sel is None else _c(sel, np.int32).reshape(-1, 3)
    n = s.shape[0]
    out = np.empty((n, block, D), dtype=np.float64)
    lse = np.empty((n, block), dtype=np.float64)
    h.oracle_masked_attention(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, Sq, Sk, D, _ptr(m), sb,
                              sh, block, None if vb is None else _ptr(vb), float(scale),
                              _ptr(s), n, _ptr(out), _ptr(lse))
    return out, lse


def vsa_forward(q_bits, k_bits, v_bits, q2k_idx, q2k_num, vbs, block: int, scale: float,
                sel=None, h=None):
    """VSA forward: LUT [B,Hq,nbq,max_kv] + counts [B,Hq,nbq] -> block mask -> masked
    attention (key blocks nbk = Sk // block)."""
    h = h or load()
    nbk = k_bits.shape[2] // block
    mask = lut_to_blockmask(q2k_idx, q2k_num, nbk, h=h)
    return masked_attention(q_bits, k_bits, v_bits, mask, block, scale, vbs=vbs, sel=sel, h=h)


def jenga_forward(q_bits, k_bits, v_bits, bitmap, block: int, scale: float, sel=None, h=None):
    """Jenga forward: i8 bitmap [nb,nb] shared by every (b,h); nonzero = attend."""
    return masked_attention(q_bits, k_bits, v_bits, bitmap, block, scale, vbs=None, sel=sel,
                            h=h)


def masked_attention_bwd(q_bits, k_bits, v_bits, dout_bits, blockmask, block: int,
                         scale: float, vbs=None, h=None):
    """Oracle backward on bf16 bit patterns (shapes as masked_attention, dout like q).
    Returns (dq [B,Hq,Sq,D], dk [B,Hkv,Sk,D], dv [B,Hkv,Sk,D]) in float64."""
    h = h or load()
    q = _c(q_bits, np.uint16)
    k = _c(k_bits, np.uint16)
    v = _c(v_bits, np.uint16)
    do = _c(dout_bits, np.uint16)
    B, Hq, Sq, D = q.shape
    Bk, Hkv, Sk, Dk = k.shape
    assert v.shape == k.shape and do.shape == q.shape and Bk == B and Dk == D
    assert Hq % Hkv == 0 and Sq % block == 0 and Sk % block == 0
    nbq, nbk = Sq // block, Sk // block
    m = _c(blockmask, np.int8)
    if m.ndim == 2:
        assert m.shape == (nbq, nbk)
        sb, sh = 0, 0
    else:
        assert m.shape == (B, Hq, nbq, nbk)
        sb, sh = Hq, 1
    vb = None if vbs is None else _c(vbs, np.int32)
    dq = np.empty((B, Hq, Sq, D), dtype=np.float64)
    dk = np.empty((B, Hkv, Sk, D), dtype=np.float64)
    dv = np.empty((B, Hkv, Sk, D), dtype=np.float64)
    h.oracle_masked_attention_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(do), B, Hq, Hkv, Sq, Sk, D,
                                  _ptr(m), sb, sh, block, None if vb is None else _ptr(vb),
                                  float(scale), _ptr(dq), _ptr(dk), _ptr(dv))
    return dq, dk, dv


def vsa_backward(q_bits, k_bits, v_bits, dout_bits, q2k_idx, q2k_num, vbs, block: int,
                 scale: float, h=None):
    """VSA backward: LUT -> block mask -> masked_attention_bwd."""
    h = h or load()
    nbk = k_bits.shape[2] // block
    mask = lut_to_blockmask(q2k_idx, q2k_num, nbk, h=h)
    return masked_attention_bwd(q_bits, k_bits, v_bits, dout_bits, mask, block, scale, vbs=vbs,
                                h=h)


def scatter_rows(out_sel, lse_sel, sel, B, H, S, block):
    """Place per-q-block results back into [B,H,S,D] / [B,H,S] arrays (NaN where not computed)."""
    D = out_sel.shape[-1]
    out = np.full((B, H, S, D), np.nan)
    lse = np.full((B, H, S), np.nan)
    for t, (b, hh, qb) in enumerate(np.asarray(sel).reshape(-1, 3)):
        out[b, hh, qb * block:(qb + 1) * block] = out_sel[t]
        lse[b, hh, qb * block:(qb + 1) * block] = lse_sel[t]
    return out, lse


if __name__ == "__main__":
    print(build(), file=sys.stderr)
