"""Thin Python binding over libvsa_gb300.so (include/vsa.h): argument marshalling only.

Every step of the forward pass and of the metadata conversions runs in the library's
CUDA kernels.  Torch is used for device memory, streams and dtype checks; there is no
CPU or eager-PyTorch fallback -- if the library is missing or was built for another
GPU the calls raise.

Functions mirror the C entry points:
  vsa_fwd, vsa_fwd_gqa, vsa_fwd_split, vsa_fwd_from_mask, jenga_fwd, vsa_bwd, vsa_lut_to_bitmap,
  vsa_bitmap_to_lut, vsa_fwd_from_host, vsa_device_status, vsa_workspace_bytes
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libvsa_gb300.so")

VSA_OK, VSA_ERR_INVALID_ARG, VSA_ERR_UNSUPPORTED, VSA_ERR_CUDA, VSA_ERR_DEVICE_TIMEOUT = range(5)
LSE_EMPTY = -3.4028234663852886e38  # -FLT_MAX, the lse of a row with no attended key
HEAD_DIM = 128
MAX_BLOCKS = 2048

# every symbol include/vsa.h declares
EXPORTS = ("vsa_fwd", "jenga_fwd", "vsa_workspace_bytes", "vsa_lut_to_bitmap",
           "vsa_bitmap_to_lut", "vsa_fwd_from_host", "vsa_device_status",
           "vsa_last_launch_count", "vsa_status_str", "vsa_fwd_noalloc", "vsa_fwd_gqa",
           "vsa_fwd_from_mask", "vsa_fwd_split", "vsa_split_workspace_bytes", "vsa_bwd",
           "vsa_bwd_workspace_bytes", "vsa_set_wait_limit_ns", "vsa_set_stall_test")
MAX_SPLITS = 64


class VsaError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} failed: {msg} (status {code})")
        self.code = code


_lib = None


def load(path: str = LIB_PATH):
    """Load the library and declare its signatures (no CUDA call happens here)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with `python -m block_sparse_attention_vsa_gb300.build`"
            " (nvcc, sm_103a); there is no fallback implementation")
    h = ctypes.CDLL(path)
    P, i32, f32, sz, u = (ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t,
                          ctypes.c_uint)
    h.vsa_fwd.restype = i32
    h.vsa_fwd.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, f32, P, P, P, P]
    h.vsa_fwd_gqa.restype = i32
    h.vsa_fwd_gqa.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32, f32, P,
                              P, P, P]
    h.vsa_fwd_split.restype = i32
    h.vsa_fwd_split.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32, f32,
                                i32, P, P, P, sz, P]
    h.vsa_split_workspace_bytes.restype = sz
    h.vsa_split_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
    h.vsa_bwd.restype = i32
    h.vsa_bwd.argtypes = [P, P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32,
                          f32, P, P, P, P, sz, P]
    h.vsa_bwd_workspace_bytes.restype = sz
    h.vsa_bwd_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
    h.vsa_fwd_from_mask.restype = i32
    h.vsa_fwd_from_mask.argtypes = [P, P, P, P, i32, P, i32, i32, i32, i32, i32, i32, i32, f32,
                                    P, P, P, P]
    h.jenga_fwd.restype = i32
    h.jenga_fwd.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, i32, f32, P, P, P, P]
    h.vsa_fwd_noalloc.restype = i32
    h.vsa_fwd_noalloc.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, f32, P, P, P]
    h.vsa_workspace_bytes.restype = sz
    h.vsa_workspace_bytes.argtypes = []
    h.vsa_lut_to_bitmap.restype = i32
    h.vsa_lut_to_bitmap.argtypes = [P, P, i32, i32, i32, P, P]
    h.vsa_bitmap_to_lut.restype = i32
    h.vsa_bitmap_to_lut.argtypes = [P, i32, i32, i32, P, P, P]
    h.vsa_fwd_from_host.restype = i32
    h.vsa_fwd_from_host.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, f32, P, P,
                                    P, P, P, P, P, P, P, P, P, P]
    h.vsa_device_status.restype = i32
    h.vsa_device_status.argtypes = [P, ctypes.POINTER(u)]
    h.vsa_last_launch_count.restype = i32
    h.vsa_last_launch_count.argtypes = []
    h.vsa_status_str.restype = ctypes.c_char_p
    h.vsa_status_str.argtypes = [i32]
    h.vsa_set_wait_limit_ns.restype = None
    h.vsa_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
    h.vsa_set_stall_test.restype = None
    h.vsa_set_stall_test.argtypes = [i32]
    _lib = h
    return h


def _check(fn: str, code: int):
    if code != VSA_OK:
        raise VsaError(fn, code, load().vsa_status_str(code).decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dev(t, name, dtype, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must be {ndim}-D, got {t.dim()}-D")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _meta32(t, name):
    """int64 metadata costs a cast (as the original wrapper does); int32 passes through."""
    if t.dtype == torch.int64:
        t = t.to(torch.int32)
    return _dev(t.contiguous(), name, torch.int32)


def workspace_bytes() -> int:
    return int(load().vsa_workspace_bytes())


def new_workspace(device=None) -> torch.Tensor:
    """A zeroed scheduling workspace; each forward call leaves it zero again."""
    n = (workspace_bytes() + 3) // 4
    return torch.zeros(n, dtype=torch.int32, device=device or "cuda")


def vsa_fwd(q, k, v, q2k_idx, q2k_num, variable_block_sizes, block=None, scale=None, out=None,
            lse=True, workspace=None, stream=None):
    """VSA forward.  q, k, v: bf16 [B,H,S,128]; q2k_idx [B,H,nb,max_kv]; q2k_num [B,H,nb];
    variable_block_sizes [nb].  Returns (out, lse or None).  ``lse`` may be True (allocate),
    False/None (skip, the inference route) or a float32 [B,H,S] tensor to write into."""
    h = load()
    _dev(q, "q", torch.bfloat16, 4)
    _dev(k, "k", torch.bfloat16, 4)
    _dev(v, "v", torch.bfloat16, 4)
    B, H, S, D = q.shape
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must have the same shape")
    vbs = _meta32(variable_block_sizes, "variable_block_sizes")
    nb = vbs.numel()
    if block is None:
        block = S // nb if nb and S % nb == 0 else 0
    idx = _meta32(q2k_idx, "q2k_idx")
    num = _meta32(q2k_num, "q2k_num")
    if idx.dim() != 4 or idx.shape[:3] != (B, H, nb) or num.shape != (B, H, nb):
        raise ValueError("q2k_idx must be [B,H,nb,max_kv] and q2k_num [B,H,nb]")
    max_kv = idx.shape[-1]
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    else:
        _dev(out, "out", torch.bfloat16, 4)
    if lse is True:
        lse_t = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    elif lse is None or lse is False:
        lse_t = None
    else:
        lse_t = _dev(lse, "lse", torch.float32, 3)
    code = h.vsa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(idx), _ptr(num), _ptr(vbs), B, H, S, D,
                     max_kv, block, scale, _ptr(out), _ptr(lse_t), _ptr(workspace),
                     _stream(stream))
    _check("vsa_fwd", code)
    return out, lse_t


def _qkv_gqa(q, k, v):
    _dev(q, "q", torch.bfloat16, 4)
    _dev(k, "k", torch.bfloat16, 4)
    _dev(v, "v", torch.bfloat16, 4)
    B, Hq, Sq, D = q.shape
    Bk, Hkv, Sk, Dk = k.shape
    if v.shape != k.shape or Bk != B or Dk != D:
        raise ValueError("k and v must be [B,Hkv,Sk,D] with q's B and D")
    return B, Hq, Hkv, Sq, Sk, D


def _lse_arg(lse, shape, device):
    if lse is True:
        return torch.empty(shape, dtype=torch.float32, device=device)
    if lse is None or lse is False:
        return None
    return _dev(lse, "lse", torch.float32, 3)


def vsa_fwd_gqa(q, k, v, q2k_idx, q2k_num, variable_block_sizes=None, block=64, scale=None,
                out=None, lse=True, workspace=None, stream=None):
    """Grouped-query / cross-length VSA forward.  q: bf16 [B,Hq,Sq,128]; k, v: bf16
    [B,Hkv,Sk,128] (Hq a multiple of Hkv); q2k_idx [B,Hq,Sq/block,max_kv] with entries in
    [0, Sk/block); q2k_num [B,Hq,Sq/block]; variable_block_sizes [Sk/block] or None."""
    h = load()
    B, Hq, Hkv, Sq, Sk, D = _qkv_gqa(q, k, v)
    idx = _meta32(q2k_idx, "q2k_idx")
    num = _meta32(q2k_num, "q2k_num")
    nbq = Sq // block if block else 0
    if idx.dim() != 4 or idx.shape[:3] != (B, Hq, nbq) or num.shape != (B, Hq, nbq):
        raise ValueError("q2k_idx must be [B,Hq,Sq/block,max_kv] and q2k_num [B,Hq,Sq/block]")
    vbs = None if variable_block_sizes is None else _meta32(variable_block_sizes,
                                                             "variable_block_sizes")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    out = torch.empty_like(q) if out is None else _dev(out, "out", torch.bfloat16, 4)
    lse_t = _lse_arg(lse, (B, Hq, Sq), q.device)
    code = h.vsa_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(idx), _ptr(num), _ptr(vbs), B, Hq, Hkv,
                         Sq, Sk, D, idx.shape[-1], block, scale, _ptr(out), _ptr(lse_t),
                         _ptr(workspace), _stream(stream))
    _check("vsa_fwd_gqa", code)
    return out, lse_t


def split_workspace_bytes(B, Hq, Sq, block, num_splits) -> int:
    return int(load().vsa_split_workspace_bytes(B, Hq, Sq, block, num_splits))


def new_split_workspace(B, Hq, Sq, block, num_splits, device=None) -> torch.Tensor:
    """Workspace for vsa_fwd_split: zeroed scheduling counters, then the partials."""
    n = split_workspace_bytes(B, Hq, Sq, block, num_splits)
    if n == 0:
        raise ValueError("invalid split-KV shape")
    return torch.zeros((n + 15) // 16 * 4, dtype=torch.int32, device=device or "cuda")


def default_splits(B, Hq, Sq, block, sm_count) -> int:
    """Ranges per item: the most that still give every (item, range) unit its own SM (1 when
    the items already fill the SMs).  One more range than that puts a few units in a second
    wave (24 heads x 98,304 keys: 6 ranges 88 us, 7 ranges 111 us), and finer ranges measured
    slower: each range pays a Q load, a pipeline fill and a 64 KB partial."""
    nbq = Sq // block
    items = B * Hq * ((nbq + 1) // 2 if block == 64 else nbq)
    if items == 0 or items >= sm_count:
        return 1
    return max(1, min(MAX_SPLITS, sm_count // items))


def vsa_fwd_split(q, k, v, q2k_idx, q2k_num, variable_block_sizes=None, block=64, scale=None,
                  num_splits=None, out=None, lse=True, workspace=None, stream=None):
    """Split-KV forward (shapes as vsa_fwd_gqa).  num_splits=None picks default_splits for
    the current device; the workspace is allocated if not given."""
    h = load()
    B, Hq, Hkv, Sq, Sk, D = _qkv_gqa(q, k, v)
    idx = _meta32(q2k_idx, "q2k_idx")
    num = _meta32(q2k_num, "q2k_num")
    nbq = Sq // block if block else 0
    if idx.dim() != 4 or idx.shape[:3] != (B, Hq, nbq) or num.shape != (B, Hq, nbq):
        raise ValueError("q2k_idx must be [B,Hq,Sq/block,max_kv] and q2k_num [B,Hq,Sq/block]")
    vbs = None if variable_block_sizes is None else _meta32(variable_block_sizes,
                                                             "variable_block_sizes")
    if num_splits is None:
        num_splits = default_splits(B, Hq, Sq, block,
                                    torch.cuda.get_device_properties(q.device).multi_processor_count)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    out = torch.empty_like(q) if out is None else _dev(out, "out", torch.bfloat16, 4)
    lse_t = _lse_arg(lse, (B, Hq, Sq), q.device)
    if workspace is None:
        workspace = new_split_workspace(B, Hq, Sq, block, num_splits, q.device)
    code = h.vsa_fwd_split(_ptr(q), _ptr(k), _ptr(v), _ptr(idx), _ptr(num), _ptr(vbs), B, Hq,
                           Hkv, Sq, Sk, D, idx.shape[-1], block, scale, num_splits, _ptr(out),
                           _ptr(lse_t), _ptr(workspace), workspace.numel() * workspace.element_size(),
                           _stream(stream))
    _check("vsa_fwd_split", code)
    return out, lse_t


def vsa_bwd(q, k, v, out, dout, lse, q2k_idx, q2k_num, variable_block_sizes=None, block=64,
            scale=None, workspace=None, stream=None):
    """Backward of vsa_fwd_gqa: returns (dq, dk, dv) for upstream gradient dout, given the
    forward's out and lse.  The workspace is allocated if not given."""
    h = load()
    B, Hq, Hkv, Sq, Sk, D = _qkv_gqa(q, k, v)
    _dev(out, "out", torch.bfloat16, 4)
    _dev(dout, "dout", torch.bfloat16, 4)
    _dev(lse, "lse", torch.float32, 3)
    idx = _meta32(q2k_idx, "q2k_idx")
    num = _meta32(q2k_num, "q2k_num")
    vbs = None if variable_block_sizes is None else _meta32(variable_block_sizes,
                                                             "variable_block_sizes")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    if workspace is None:
        n = int(h.vsa_bwd_workspace_bytes(B, Hq, Sq, Sk, block))
        workspace = torch.empty(max(n, 1), dtype=torch.uint8, device=q.device)
    code = h.vsa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(idx),
                     _ptr(num), _ptr(vbs), B, Hq, Hkv, Sq, Sk, D, idx.shape[-1], block, scale,
                     _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
                     workspace.numel() * workspace.element_size(), _stream(stream))
    _check("vsa_bwd", code)
    return dq, dk, dv


def vsa_fwd_from_mask(q, k, v, block_map, variable_block_sizes=None, block=64, scale=None,
                      out=None, lse=True, workspace=None, stream=None):
    """Forward from a block map: bool/int8 [B,Hq,Sq/block,Sk/block] (one per query head) or
    [Sq/block,Sk/block] (shared by every head).  Shapes otherwise as vsa_fwd_gqa."""
    h = load()
    B, Hq, Hkv, Sq, Sk, D = _qkv_gqa(q, k, v)
    if block_map.dtype == torch.bool:
        block_map = block_map.to(torch.int8)
    _dev(block_map, "block_map", torch.int8)
    nbq, nbk = (Sq // block, Sk // block) if block else (0, 0)
    if tuple(block_map.shape) == (nbq, nbk):
        shared = 1
    elif tuple(block_map.shape) == (B, Hq, nbq, nbk):
        shared = 0
    else:
        raise ValueError("block_map must be [B,Hq,Sq/block,Sk/block] or [Sq/block,Sk/block]")
    vbs = None if variable_block_sizes is None else _meta32(variable_block_sizes,
                                                             "variable_block_sizes")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    out = torch.empty_like(q) if out is None else _dev(out, "out", torch.bfloat16, 4)
    lse_t = _lse_arg(lse, (B, Hq, Sq), q.device)
    code = h.vsa_fwd_from_mask(_ptr(q), _ptr(k), _ptr(v), _ptr(block_map), shared, _ptr(vbs), B,
                               Hq, Hkv, Sq, Sk, D, block, scale, _ptr(out), _ptr(lse_t),
                               _ptr(workspace), _stream(stream))
    _check("vsa_fwd_from_mask", code)
    return out, lse_t


def vsa_fwd_noalloc(q, k, v, q2k_idx, q2k_num, variable_block_sizes, block=None, scale=None,
                    out=None, lse=None, stream=None):
    """vsa_fwd for callers that cannot hand the library any device memory of their own:
    the scheduling scratch lives in a static array inside the library (shared by every
    call on the device, so calls must not overlap on the GPU).  ``out`` and ``lse`` must
    be given when the caller cannot allocate (they are allocated here only if omitted).
    Returns (out, lse or None)."""
    h = load()
    _dev(q, "q", torch.bfloat16, 4)
    B, H, S, D = q.shape
    vbs = _meta32(variable_block_sizes, "variable_block_sizes")
    nb = vbs.numel()
    if block is None:
        block = S // nb if nb and S % nb == 0 else 0
    idx = _meta32(q2k_idx, "q2k_idx")
    num = _meta32(q2k_num, "q2k_num")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    code = h.vsa_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(idx), _ptr(num), _ptr(vbs), B, H,
                             S, D, idx.shape[-1], block, scale, _ptr(out), _ptr(lse),
                             _stream(stream))
    _check("vsa_fwd_noalloc", code)
    return out, lse


def jenga_fwd(q, k, v, mask_bitmap, block_q=64, block_k=64, scale=None, out=None, lse=True,
              workspace=None, stream=None):
    """Jenga forward from an i8 bitmap [S/block_q, S/block_k] shared by every (b, h)."""
    h = load()
    _dev(q, "q", torch.bfloat16, 4)
    _dev(k, "k", torch.bfloat16, 4)
    _dev(v, "v", torch.bfloat16, 4)
    B, H, S, D = q.shape
    if mask_bitmap.dtype == torch.bool:
        mask_bitmap = mask_bitmap.to(torch.int8)
    _dev(mask_bitmap, "mask_bitmap", torch.int8, 2)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    if lse is True:
        lse_t = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    elif lse is None or lse is False:
        lse_t = None
    else:
        lse_t = _dev(lse, "lse", torch.float32, 3)
    code = h.jenga_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(mask_bitmap), B, H, S, D, block_q,
                       block_k, scale, _ptr(out), _ptr(lse_t), _ptr(workspace), _stream(stream))
    _check("jenga_fwd", code)
    return out, lse_t


def vsa_lut_to_bitmap(q2k_idx, q2k_num, nb, stream=None):
    """[..., rows, max_kv] + [..., rows] -> int8 [..., rows, nb] (bit-exact 0/1)."""
    h = load()
    idx = _meta32(q2k_idx, "q2k_idx")
    num = _meta32(q2k_num, "q2k_num")
    max_kv = idx.shape[-1]
    rows = num.numel()
    out = torch.empty(tuple(num.shape) + (nb,), dtype=torch.int8, device=idx.device)
    _check("vsa_lut_to_bitmap",
           h.vsa_lut_to_bitmap(_ptr(idx), _ptr(num), rows, max_kv, nb, _ptr(out), _stream(stream)))
    return out


def vsa_bitmap_to_lut(bitmap, max_kv, stream=None):
    """int8 [..., rows, nb] -> (int32 [..., rows, max_kv] ascending, -1 padded; int32 [..., rows])."""
    h = load()
    if bitmap.dtype == torch.bool:
        bitmap = bitmap.to(torch.int8)
    _dev(bitmap, "bitmap", torch.int8)
    nb = bitmap.shape[-1]
    rows = bitmap.numel() // nb
    idx = torch.empty(tuple(bitmap.shape[:-1]) + (max_kv,), dtype=torch.int32, device=bitmap.device)
    num = torch.empty(tuple(bitmap.shape[:-1]), dtype=torch.int32, device=bitmap.device)
    _check("vsa_bitmap_to_lut",
           h.vsa_bitmap_to_lut(_ptr(bitmap), rows, nb, max_kv, _ptr(idx), _ptr(num),
                               _stream(stream)))
    return idx, num


def vsa_fwd_from_host(h_q, h_k, h_v, h_idx, h_num, h_vbs, block, scale, h_out, h_lse, dev_bufs,
                      workspace=None, stream=None):
    """Host-buffer entry: copies in, runs vsa_fwd, copies out -- all enqueued on ``stream``.
    ``dev_bufs`` = dict of device tensors q, k, v, idx, num, vbs, out, lse (lse may be None)."""
    h = load()
    B, H, S, D = h_q.shape
    max_kv = h_idx.shape[-1]
    d = dev_bufs
    code = h.vsa_fwd_from_host(_ptr(h_q), _ptr(h_k), _ptr(h_v), _ptr(h_idx), _ptr(h_num),
                               _ptr(h_vbs), B, H, S, D, max_kv, block, float(scale), _ptr(h_out),
                               _ptr(h_lse), _ptr(d["q"]), _ptr(d["k"]), _ptr(d["v"]),
                               _ptr(d["idx"]), _ptr(d["num"]), _ptr(d["vbs"]), _ptr(d["out"]),
                               _ptr(d.get("lse")), _ptr(workspace), _stream(stream))
    _check("vsa_fwd_from_host", code)


def vsa_device_status(stream=None):
    """(status code, detail) of the device status word; synchronises the stream."""
    h = load()
    detail = ctypes.c_uint(0)
    code = h.vsa_device_status(_stream(stream), ctypes.byref(detail))
    return code, detail.value


def vsa_last_launch_count() -> int:
    return int(load().vsa_last_launch_count())


def vsa_set_wait_limit_ns(ns: int) -> None:
    """Timeout-path test hook: limit of the kernels' non-drain waits (0 = the full limit)."""
    load().vsa_set_wait_limit_ns(int(ns))


def vsa_set_stall_test(enable: bool) -> None:
    """Timeout-path test hook: while on, every launch's MMA warp waits on a barrier nothing
    completes, so the launch reports VSA_ERR_DEVICE_TIMEOUT."""
    load().vsa_set_stall_test(1 if enable else 0)
