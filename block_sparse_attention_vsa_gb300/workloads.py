"""Seeded synthetic inputs shaped like the workloads block-sparse VSA / Jenga attention
is measured on.

This module only draws random numbers and lays out index structure.  It holds
none of the attention arithmetic, imports neither the CUDA binding nor the
oracle, and is the one piece of code that both sides of every parity test use.

Recipe (every workload, seed 0 unless a test says otherwise), all on the CPU with
one ``torch.Generator``:
  1. q, k, v = randn([B, H, S, 128], fp32), drawn in that order; for the Jenga
     workload q and k are multiplied by 3 in fp32 (a peaky softmax);
  2. each is rounded to bf16 (round-to-nearest-even);
  3. the block metadata is drawn next from the same generator.

The five workloads:
  vsa_tiny        B1 H1 S512 block 64 (8 blocks); q2k_num ~ U{0..8} (0 included);
                  q2k_idx distinct random, ascending, pad -1; all blocks full (64)
  vsa_mid         B1 H12 S16384 block 64 (256 blocks); every q-block takes its own
                  diagonal block plus 63 distinct random others (25 %)
  vsa_blk128      B2 H24 S32768 block 128 (256 blocks); q2k_num ~ U{1..51}
                  distinct random blocks; variable_block_sizes ~ U{96..128}
  jenga           B1 H16 S24576, 64x64 blocks, one i8 bitmap [384, 384] shared by
                  every head: the band kb - qb in [-8, 7] plus 8 distinct random
                  blocks outside the band per row
  vsa_decode      B1 H24, 128 queries (one block-64 pair per head) against 98304 keys
                  (1536 blocks): each query block takes 128 distinct random key blocks;
                  variable_block_sizes 64 except the last block, 32 (a short query
                  over a long video context, run through the split-KV path)
  vsa_long_video  B1 H24 S98304 block 64 (1536 blocks) on a 16x16x6 block grid,
                  id = (x*16 + y)*6 + z; every q-block takes the 112 blocks nearest
                  to it (squared Euclidean distance, ties by id, itself included)
                  plus 16 distinct random others (128 = 8.3 %);
                  variable_block_sizes 64 except the last block, 32

Grouped-query / cross-length and block-map cases (make_random_gqa) draw q as
[B, Hq, Sq, 128] and k, v as [B, Hkv, Sk, 128] in the same order and way; their LUT
rows pick distinct random key blocks of [0, Sk/block), and the block-map form is the
0/1 expansion of those rows (one int8 map per (b, hq)).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

HEAD_DIM = 128


@dataclass
class Workload:
    name: str
    kind: str                      # "vsa" or "jenga"
    B: int
    H: int
    S: int
    D: int
    block: int
    scale: float
    q: torch.Tensor                # bf16 [B,H,S,D], CPU
    k: torch.Tensor
    v: torch.Tensor
    q2k_idx: np.ndarray | None = None   # int32 [B,H,nb,max_kv]
    q2k_num: np.ndarray | None = None   # int32 [B,H,nb]
    vbs: np.ndarray | None = None       # int32 [nb]
    bitmap: np.ndarray | None = None    # int8 [nb,nb] (jenga)
    extra: dict = field(default_factory=dict)
    Hkv: int | None = None              # key/value heads (None = H)
    Sk: int | None = None               # key length (None = S)
    block_map: np.ndarray | None = None  # int8 [B,H,nbq,nbk] or [nbq,nbk] ("mask" kind)

    def __post_init__(self):
        if self.Hkv is None:
            self.Hkv = self.H
        if self.Sk is None:
            self.Sk = self.S

    @property
    def nb(self) -> int:
        return self.S // self.block

    @property
    def nbq(self) -> int:
        return self.S // self.block

    @property
    def nbk(self) -> int:
        return self.Sk // self.block

    @property
    def max_kv(self) -> int:
        return 0 if self.q2k_idx is None else int(self.q2k_idx.shape[-1])


SPECS = {
    "vsa_tiny": dict(kind="vsa", B=1, H=1, S=512, block=64),
    "vsa_mid": dict(kind="vsa", B=1, H=12, S=16384, block=64),
    "vsa_blk128": dict(kind="vsa", B=2, H=24, S=32768, block=128),
    "jenga": dict(kind="jenga", B=1, H=16, S=24576, block=64),
    "vsa_long_video": dict(kind="vsa", B=1, H=24, S=98304, block=64),
}


def gen(seed: int = 0) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(seed)
    return g


def randn_bf16(shape, g: torch.Generator, mul: float = 1.0) -> torch.Tensor:
    """N(0,1) in fp32 (optionally times ``mul`` in fp32), rounded to bf16."""
    x = torch.randn(shape, generator=g, dtype=torch.float32)
    if mul != 1.0:
        x.mul_(mul)
    y = x.to(torch.bfloat16)
    del x
    return y


def make_qkv(B, H, S, D, g, mul_qk: float = 1.0):
    q = randn_bf16((B, H, S, D), g, mul_qk)
    k = randn_bf16((B, H, S, D), g, mul_qk)
    v = randn_bf16((B, H, S, D), g)
    return q, k, v


def _rows_from_ranks(rank_keys: torch.Tensor, counts: torch.Tensor, max_kv: int) -> np.ndarray:
    """Pick, per row, the ``counts[row]`` entries with the smallest key, write them
    ascending into a [.., max_kv] row and pad with -1."""
    order = torch.argsort(rank_keys, dim=-1)[..., :max_kv]
    big = rank_keys.shape[-1] + 1
    if order.shape[-1] < max_kv:
        pad = torch.full(order.shape[:-1] + (max_kv - order.shape[-1],), big, dtype=order.dtype)
        order = torch.cat([order, pad], dim=-1)
    slot = torch.arange(max_kv).expand_as(order)
    chosen = torch.where(slot < counts.unsqueeze(-1), order, torch.full_like(order, big))
    chosen, _ = torch.sort(chosen, dim=-1)
    chosen = torch.where(chosen == big, torch.full_like(chosen, -1), chosen)
    return chosen.to(torch.int32).numpy()


def random_lut(B, H, nb, max_kv, g, n_lo, n_hi, force_diag=False):
    """Distinct random blocks per row, ascending, -1 padded; counts ~ U{n_lo..n_hi}."""
    counts = torch.randint(n_lo, n_hi + 1, (B, H, nb), generator=g)
    keys = torch.rand((B, H, nb, nb), generator=g)
    if force_diag:
        eye = torch.eye(nb, dtype=torch.bool).expand(B, H, nb, nb)
        keys = torch.where(eye, torch.full_like(keys, -1.0), keys)
    idx = _rows_from_ranks(keys, counts, max_kv)
    return idx, counts.to(torch.int32).numpy()


def make_vsa_tiny(seed=0) -> Workload:
    B, H, S, D, block = 1, 1, 512, HEAD_DIM, 64
    nb = S // block
    g = gen(seed)
    q, k, v = make_qkv(B, H, S, D, g)
    idx, num = random_lut(B, H, nb, 8, g, 0, 8)
    vbs = np.full(nb, block, dtype=np.int32)
    return Workload("vsa_tiny", "vsa", B, H, S, D, block, 1.0 / math.sqrt(D), q, k, v,
                    q2k_idx=idx, q2k_num=num, vbs=vbs)


def make_vsa_mid(seed=0) -> Workload:
    B, H, S, D, block = 1, 12, 16384, HEAD_DIM, 64
    nb = S // block
    g = gen(seed)
    q, k, v = make_qkv(B, H, S, D, g)
    idx, num = random_lut(B, H, nb, 64, g, 64, 64, force_diag=True)
    vbs = np.full(nb, block, dtype=np.int32)
    return Workload("vsa_mid", "vsa", B, H, S, D, block, 1.0 / math.sqrt(D), q, k, v,
                    q2k_idx=idx, q2k_num=num, vbs=vbs)


def make_vsa_blk128(seed=0) -> Workload:
    B, H, S, D, block = 2, 24, 32768, HEAD_DIM, 128
    nb = S // block
    g = gen(seed)
    q, k, v = make_qkv(B, H, S, D, g)
    idx, num = random_lut(B, H, nb, 51, g, 1, 51)
    vbs = torch.randint(96, 129, (nb,), generator=g).to(torch.int32).numpy()
    return Workload("vsa_blk128", "vsa", B, H, S, D, block, 1.0 / math.sqrt(D), q, k, v,
                    q2k_idx=idx, q2k_num=num, vbs=vbs)


def jenga_bitmap(nb: int, g: torch.Generator, lo=-8, hi=7, extra=8) -> np.ndarray:
    qb = torch.arange(nb).unsqueeze(1)
    kb = torch.arange(nb).unsqueeze(0)
    band = ((kb - qb) >= lo) & ((kb - qb) <= hi)
    keys = torch.rand((nb, nb), generator=g)
    keys = torch.where(band, torch.full_like(keys, 2.0), keys)
    pick = torch.argsort(keys, dim=-1)[:, :extra]
    bm = band.clone()
    bm.scatter_(1, pick, True)
    return bm.to(torch.int8).numpy()


def make_jenga(seed=0) -> Workload:
    B, H, S, D, block = 1, 16, 24576, HEAD_DIM, 64
    nb = S // block
    g = gen(seed)
    q, k, v = make_qkv(B, H, S, D, g, mul_qk=3.0)
    bm = jenga_bitmap(nb, g)
    return Workload("jenga", "jenga", B, H, S, D, block, 1.0 / math.sqrt(D), q, k, v,
                    bitmap=bm)


def grid_neighbours(gx: int, gy: int, gz: int, n_near: int) -> np.ndarray:
    """For every block id = (x*gy + y)*gz + z of a gx*gy*gz grid, the ids of the
    ``n_near`` nearest blocks (squared Euclidean distance, ties by id), itself included."""
    ids = np.arange(gx * gy * gz)
    x, y, z = ids // (gy * gz), (ids // gz) % gy, ids % gz
    d2 = ((x[:, None] - x[None, :]) ** 2 + (y[:, None] - y[None, :]) ** 2
          + (z[:, None] - z[None, :]) ** 2)
    n = ids.size
    key = d2.astype(np.int64) * n + ids[None, :]
    return np.argsort(key, axis=1, kind="stable")[:, :n_near].astype(np.int64)


def make_vsa_long_video(seed=0, H=24) -> Workload:
    B, S, D, block = 1, 98304, HEAD_DIM, 64
    nb = S // block
    g = gen(seed)
    q, k, v = make_qkv(B, H, S, D, g)
    near = torch.from_numpy(grid_neighbours(16, 16, 6, 112))          # [nb,112]
    keys = torch.rand((B, H, nb, nb), generator=g)
    keys.scatter_(-1, near.expand(B, H, nb, 112).contiguous(), 2.0)
    extra = torch.argsort(keys, dim=-1)[..., :16]
    del keys
    rows = torch.cat([near.expand(B, H, nb, 112), extra], dim=-1)
    rows, _ = torch.sort(rows, dim=-1)
    idx = rows.to(torch.int32).numpy()
    num = np.full((B, H, nb), 128, dtype=np.int32)
    vbs = np.full(nb, block, dtype=np.int32)
    vbs[-1] = 32
    return Workload("vsa_long_video", "vsa", B, H, S, D, block, 1.0 / math.sqrt(D), q, k, v,
                    q2k_idx=idx, q2k_num=num, vbs=vbs)


def make_vsa_decode(seed=0) -> Workload:
    B, H, Sq, Sk, D, block = 1, 24, 128, 98304, HEAD_DIM, 64
    w = make_random_gqa(B, H, H, Sq, Sk, D, block, 128, seed, n_lo=128, n_hi=128)
    w.vbs = np.full(Sk // block, block, dtype=np.int32)
    w.vbs[-1] = 32
    w.name = "vsa_decode"
    return w


MAKERS = {
    "vsa_tiny": make_vsa_tiny,
    "vsa_mid": make_vsa_mid,
    "vsa_blk128": make_vsa_blk128,
    "jenga": make_jenga,
    "vsa_long_video": make_vsa_long_video,
    "vsa_decode": make_vsa_decode,
}


def make(name: str, seed: int = 0) -> Workload:
    return MAKERS[name](seed)


def make_random_vsa(B, H, S, D, block, max_kv, seed, n_lo=0, n_hi=None, vbs_lo=None,
                    vbs_hi=None, qk_mul=1.0) -> Workload:
    """A small VSA case for parity tests: distinct random blocks, counts ~ U{n_lo..n_hi},
    variable_block_sizes ~ U{vbs_lo..vbs_hi} (default: full blocks)."""
    nb = S // block
    n_hi = min(max_kv, nb) if n_hi is None else n_hi
    g = gen(seed)
    q, k, v = make_qkv(B, H, S, D, g, mul_qk=qk_mul)
    idx, num = random_lut(B, H, nb, max_kv, g, n_lo, n_hi)
    if vbs_lo is None:
        vbs = np.full(nb, block, dtype=np.int32)
    else:
        vbs = torch.randint(vbs_lo, vbs_hi + 1, (nb,), generator=g).to(torch.int32).numpy()
    return Workload("random_vsa", "vsa", B, H, S, D, block, 1.0 / math.sqrt(D), q, k, v,
                    q2k_idx=idx, q2k_num=num, vbs=vbs)


def make_random_gqa(B, Hq, Hkv, Sq, Sk, D, block, max_kv, seed, n_lo=0, n_hi=None,
                    vbs_lo=None, vbs_hi=None, kind="vsa", shared_map=False,
                    qk_mul=1.0) -> Workload:
    """Grouped-query / cross-length case: q [B,Hq,Sq,D], k and v [B,Hkv,Sk,D].  kind "vsa"
    carries the LUT (rows over the Sk/block key blocks); kind "mask" carries the same
    selection as an int8 block map [B,Hq,nbq,nbk], or with ``shared_map`` the map of
    (b=0, hq=0) alone as [nbq,nbk] for every head."""
    nbq, nbk = Sq // block, Sk // block
    n_hi = min(max_kv, nbk) if n_hi is None else n_hi
    g = gen(seed)
    q = randn_bf16((B, Hq, Sq, D), g, qk_mul)
    k = randn_bf16((B, Hkv, Sk, D), g, qk_mul)
    v = randn_bf16((B, Hkv, Sk, D), g)
    counts = torch.randint(n_lo, n_hi + 1, (B, Hq, nbq), generator=g)
    keys = torch.rand((B, Hq, nbq, max(nbk, 1)), generator=g)[..., :nbk]
    idx = _rows_from_ranks(keys, counts, max_kv)
    num = counts.to(torch.int32).numpy()
    if vbs_lo is None:
        vbs = np.full(nbk, block, dtype=np.int32)
    else:
        vbs = torch.randint(vbs_lo, vbs_hi + 1, (nbk,), generator=g).to(torch.int32).numpy()
    w = Workload("random_gqa", kind, B, Hq, Sq, D, block, 1.0 / math.sqrt(D), q, k, v,
                 q2k_idx=idx, q2k_num=num, vbs=vbs, Hkv=Hkv, Sk=Sk)
    if kind == "mask":
        bm = np.zeros((B, Hq, nbq, nbk), dtype=np.int8)
        slot = np.arange(max_kv)
        for b in range(B):
            for h in range(Hq):
                for qb in range(nbq):
                    row = idx[b, h, qb][slot < num[b, h, qb]]
                    bm[b, h, qb, row] = 1
        w.block_map = np.ascontiguousarray(bm[0, 0]) if shared_map else bm
    return w


def first_heads(w: Workload, n: int) -> Workload:
    """The same workload restricted to its first ``n`` query heads (and their key/value
    heads): every per-head structure is unchanged, only the head count shrinks."""
    n = max(1, min(n, w.H))
    group = w.H // w.Hkv
    nkv = max(1, n // group)
    out = Workload(f"{w.name}_h{n}", w.kind, w.B, n, w.S, w.D, w.block, w.scale,
                   w.q[:, :n].contiguous(), w.k[:, :nkv].contiguous(),
                   w.v[:, :nkv].contiguous(), bitmap=w.bitmap, extra=dict(w.extra),
                   Hkv=nkv, Sk=w.Sk)
    if w.q2k_idx is not None:
        out.q2k_idx = np.ascontiguousarray(w.q2k_idx[:, :n])
        out.q2k_num = np.ascontiguousarray(w.q2k_num[:, :n])
    out.vbs = w.vbs
    if w.block_map is not None:
        out.block_map = w.block_map if w.block_map.ndim == 2 else np.ascontiguousarray(
            w.block_map[:, :n])
    return out


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> its uint16 bit patterns (a view, no rounding)."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)
