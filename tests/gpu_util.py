"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI and the
oracle on the same seeded inputs, compare with the tolerances of the contract.

Tolerances (bf16 inputs and output, fp32 accumulation; the oracle is fp64):
  out: max |gpu - oracle| <= 2e-2 and mean |gpu - oracle| <= 2e-3
  lse: max |gpu - oracle| <= 1e-3
  rows with no attended key: out exactly +0 and lse exactly the sentinel on both sides.
"""
import numpy as np
import torch

from block_sparse_attention_vsa_gb300 import binding, workloads
from oracle import oracle as orc

OUT_MAX, OUT_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3


def to_dev(w):
    d = torch.device("cuda:0")
    r = dict(q=w.q.to(d), k=w.k.to(d), v=w.v.to(d))
    if w.kind == "vsa":
        r["idx"] = torch.from_numpy(np.ascontiguousarray(w.q2k_idx)).to(d)
        r["num"] = torch.from_numpy(np.ascontiguousarray(w.q2k_num)).to(d)
        r["vbs"] = torch.from_numpy(np.ascontiguousarray(w.vbs)).to(d)
    elif w.kind == "mask":
        r["map"] = torch.from_numpy(np.ascontiguousarray(w.block_map)).to(d)
        r["vbs"] = torch.from_numpy(np.ascontiguousarray(w.vbs)).to(d)
    else:
        r["bitmap"] = torch.from_numpy(np.ascontiguousarray(w.bitmap)).to(d)
    return r


def run_gpu(w, dev=None, lse=True, workspace=None, splits=None):
    dev = dev or to_dev(w)
    gqa = w.Hkv != w.H or w.Sk != w.S
    if splits is not None:
        out, l = binding.vsa_fwd_split(dev["q"], dev["k"], dev["v"], dev["idx"], dev["num"],
                                       dev["vbs"], block=w.block, scale=w.scale,
                                       num_splits=splits, lse=lse, workspace=workspace)
    elif w.kind == "vsa" and gqa:
        out, l = binding.vsa_fwd_gqa(dev["q"], dev["k"], dev["v"], dev["idx"], dev["num"],
                                     dev["vbs"], block=w.block, scale=w.scale, lse=lse,
                                     workspace=workspace)
    elif w.kind == "mask":
        out, l = binding.vsa_fwd_from_mask(dev["q"], dev["k"], dev["v"], dev["map"], dev["vbs"],
                                           block=w.block, scale=w.scale, lse=lse,
                                           workspace=workspace)
    elif w.kind == "vsa":
        out, l = binding.vsa_fwd(dev["q"], dev["k"], dev["v"], dev["idx"], dev["num"], dev["vbs"],
                                 block=w.block, scale=w.scale, lse=lse, workspace=workspace)
    else:
        out, l = binding.jenga_fwd(dev["q"], dev["k"], dev["v"], dev["bitmap"], w.block, w.block,
                                   scale=w.scale, lse=lse, workspace=workspace)
    torch.cuda.synchronize()
    code, detail = binding.vsa_device_status()
    assert code == binding.VSA_OK, f"device status {code}, detail {detail:#x}"
    return out, l


def run_oracle(w, sel=None):
    qb, kb, vb = workloads.bits(w.q), workloads.bits(w.k), workloads.bits(w.v)
    if w.kind == "vsa":
        return orc.vsa_forward(qb, kb, vb, w.q2k_idx, w.q2k_num, w.vbs, w.block, w.scale, sel=sel)
    if w.kind == "mask":
        return orc.masked_attention(qb, kb, vb, w.block_map, w.block, w.scale, vbs=w.vbs,
                                    sel=sel)
    return orc.jenga_forward(qb, kb, vb, w.bitmap, w.block, w.scale, sel=sel)


def gather_rows(t, sel, block):
    """[B,H,S,...] device tensor -> numpy rows of the selected q-blocks, [n, block, ...]."""
    a = t.float().cpu().numpy()
    return np.stack([a[b, h, qb * block:(qb + 1) * block] for (b, h, qb) in sel])


def compare(w, out, lse, sel=None):
    sel = orc.all_qblocks(w.B, w.H, w.nbq) if sel is None else np.asarray(sel, np.int32)
    ref_o, ref_l = run_oracle(w, sel)
    o = gather_rows(out, sel, w.block).astype(np.float64)
    err = np.abs(o - ref_o)
    stats = dict(out_max=float(err.max()), out_mean=float(err.mean()))
    assert err.max() <= OUT_MAX and err.mean() <= OUT_MEAN, stats
    empty = ref_l == orc.LSE_EMPTY
    if empty.any():
        assert np.all(o[empty] == 0.0) and not np.any(np.signbit(o[empty])), "empty rows not +0"
    if lse is not None:
        l = gather_rows(lse, sel, w.block).astype(np.float64)
        if empty.any():
            assert np.all(l[empty] == orc.LSE_EMPTY), "empty rows: lse not the sentinel"
        lerr = np.abs(l[~empty] - ref_l[~empty]) if (~empty).any() else np.zeros(1)
        stats["lse_max"] = float(lerr.max())
        assert lerr.max() <= LSE_MAX, stats
    return stats


def sample_qblocks(B, H, nb, per_head, seed, must=()):
    """Seeded sample of q-blocks per (b, h): always 0 and nb-1 plus ``must``, then random."""
    rng = np.random.default_rng(seed)
    sel = []
    for b in range(B):
        for h in range(H):
            pick = {0, nb - 1} | set(int(x) for x in must)
            pool = [x for x in range(nb) if x not in pick]
            extra = rng.choice(pool, size=max(0, per_head - len(pick)), replace=False)
            for qb in sorted(pick | set(int(x) for x in extra)):
                sel.append((b, h, qb))
    return np.array(sel, np.int32)
