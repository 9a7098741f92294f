// vsa_bwd_kernel.cuh -- backward of the block-sparse attention forward (dq, dk, dv).
//
// What it computes: the gradient of the forward of vsa_fwd_kernel.cuh for a given dout,
// over the attended keys only ("FastVideo block_sparse_attn_sm100a.py", module docstring:
// the backward consumes the forward's base-2 lse):
//   p_ij  = 2^(s_ij * scale * log2 e - lse_i)   (0 for masked keys and empty rows)
//   D_i   = dout_i . out_i
//   ds_ij = p_ij (dout_i . v_j - D_i)
//   dq_i  = scale sum_j ds_ij k_j,   dk_j = scale sum_i ds_ij q_i,   dv_j = sum_i p_ij dout_i
// with dk and dv summed over every query head of a key/value group.
//
// Kernels:
//   bwd_prep_kernel   per query row, one warp each: -D_i, and -lse_i (-inf for a row that
//                     attends no key, so that every p of the row comes out 0).
//   bsa_bwd_kernel    one CTA per (batch, key/value head, key tile of 128 keys): a tile is
//                     one key block (block 128) or an adjacent pair of key blocks (block
//                     64).  K and V of the tile stay in SMEM and dK, dV accumulate in TMEM
//                     while the CTA walks the (query head of the group, query block) pairs
//                     selecting the tile -- a column of the 0/1 block map, compacted into
//                     an SMEM list -- 64 query rows a step (two steps per block-128 query
//                     block, one per block-64 query block).  A block-64 pair walks the
//                     union of the query blocks selecting either of its key blocks; each
//                     list entry says which of the two it selects, and the keys of the
//                     other are masked.  With neighbourhood selections, where adjacent key
//                     blocks are selected by mostly the same query blocks, the pair loads
//                     each shared query block's Q/dO and reduces its dQ once instead of
//                     twice.  Per step, on the 5th-generation tensor cores:
//                       S^T  = K Q^T      (M = 128 keys, N = 64 queries, K = d) -> TMEM
//                       dP^T = V dO^T                                           -> TMEM
//                       P^T, dS^T formed by the gradient warps (one thread per key row);
//                       P^T written back over S^T in TMEM as bf16, dS^T to SMEM (without
//                       the factor scale, which the dK epilogue and bwd_dq_kernel apply)
//                       dV  += P^T dO     (A = P^T from TMEM, B = dO MN-major)
//                       dK  += dS^T Q     (A = dS^T K-major in SMEM, B = Q MN-major)
//                       dQ^T = K^T dS^T   (both operands MN-major in SMEM; M = 128 d)
//                     and the dQ warps add dQ^T (one thread per d column, 64 query rows)
//                     into an fp32 accumulator with coalesced reductions: several key blocks
//                     feed every query row.
//   bwd_dq_kernel     fp32 dQ accumulator times scale -> bf16 dq.
//
// bsa_bwd_kernel roles (15 warps):
//   warps 0-7   gradient warps: warpgroup w handles query columns 32w..32w+31 of a step,
//               thread = key row (TMEM lane); after the last step they store dV (warps
//               0-3) and dK (warps 4-7) as bf16.
//   warps 8-11  dQ warps: thread = d column (TMEM lane of dQ^T).
//   warp 12     TMA: K, V once; per step Q, dO (64 rows) and -lse, -D (64 floats) into a
//               3-stage ring.
//   warp 13     MMA issuer of S^T, dP^T, dV; owns the TMEM allocation.
//   warp 14     list: compacts the block-map column into the step list (in chunks);
//               during the steps it issues the dK and dQ^T MMAs (a second issuing
//               thread: they depend on no other MMA of the step).
//               Both issuing warps run their loops converged and the lane elect.sync
//               picks issues (predicated, not branched): half the issue time per MMA.
// TMEM (512 columns): two step slots (step g uses slot g & 1) at 0 and 128, each holding
// S^T in its first 64 columns (P^T bf16 over 0-15 and 32-47) and dP^T in the next 64 (then
// dQ^T of the same step, written over the consumed dP^T); dV 256-383, dK 384-511.  dS^T
// lives in SMEM only, one tile per slot.
// MMA issue order on warp 13: S_0, dP_0, then per step t: S_{t+1}, dV_t, dP_{t+1}, so the
// next step's S^T is computed while the gradient warps form P^T and dS^T of this one.
// tcgen05 MMAs of one thread execute in issue order: S_{t+2} lands in the slot whose P^T dV_t
// read.  dP_{t+1} waits until the dQ warps have read dQ^T of step t - 1 out of its columns.
// dK_t and dQ_t, on warp 14, are ordered by barriers alone: they wait for dS^T of step t
// (which comes after the gradient warps read dP^T_t), and the gradient warps overwrite a
// slot's SMEM dS^T only after dQ_{t-2} (issued after dK_{t-2}) has completed.  The Q/dO
// stage of a step is free once both threads' readers are done.
// Every mbarrier wait is bounded; a wait that runs out records a code in the device
// status word, raises the CTA's abort flag and every role returns.
#pragma once

#include <cuda.h>

#include <cstdint>

#include "sm103_ptx.cuh"

namespace vsa {

// For rows rows, one warp per row (4 elements per lane): nD[i] = -sum_d dout[i][d] out[i][d]
// and nlse[i] = -lse[i], or -inf where lse[i] is -inf (a row that attends no key).
__global__ void __launch_bounds__(256) bwd_prep_kernel(const uint16_t* __restrict__ out,
                                                       const uint16_t* __restrict__ dout,
                                                       const float* __restrict__ lse,
                                                       long long rows, float* __restrict__ nD,
                                                       float* __restrict__ nlse) {
  const long long r = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (r >= rows) return;
  const uint32_t lane = threadIdx.x & 31;
  const uint2 o = reinterpret_cast<const uint2*>(out + r * 128)[lane];
  const uint2 g = reinterpret_cast<const uint2*>(dout + r * 128)[lane];
  float acc = 0.0f;
  const uint32_t ow[2] = {o.x, o.y}, gw[2] = {g.x, g.y};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    acc = fmaf(__uint_as_float(ow[i] << 16), __uint_as_float(gw[i] << 16), acc);
    acc = fmaf(__uint_as_float(ow[i] & 0xFFFF0000u), __uint_as_float(gw[i] & 0xFFFF0000u), acc);
  }
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
  if (lane == 0) {
    nD[r] = -acc;
    const float l = lse[r];
    nlse[r] = l > -3.0e38f ? -l : -INFINITY;
  }
}

// scale times the fp32 dQ accumulator -> bf16 (round to nearest even), 8 elements per thread.
__global__ void __launch_bounds__(256) bwd_dq_kernel(const float* __restrict__ acc,
                                                     long long n8, float scale,
                                                     uint16_t* __restrict__ dq) {
  const long long i = (long long)blockIdx.x * 256 + threadIdx.x;
  if (i >= n8) return;
  const float4 a = reinterpret_cast<const float4*>(acc)[2 * i];
  const float4 b = reinterpret_cast<const float4*>(acc)[2 * i + 1];
  uint4 o;
  o.x = pack_bf16x2(a.x * scale, a.y * scale);
  o.y = pack_bf16x2(a.z * scale, a.w * scale);
  o.z = pack_bf16x2(b.x * scale, b.y * scale);
  o.w = pack_bf16x2(b.z * scale, b.w * scale);
  reinterpret_cast<uint4*>(dq)[i] = o;
}

struct BwdArgs {
  const float* nlse;        // [B*Hq*Sq] -lse (base 2), -inf for a row that attends no key
  const float* nD;          // [B*Hq*Sq] -D
  const int8_t* bitmap;     // [B*Hq*nbq, nbk] 0/1 block map
  const int32_t* vbs;       // [nbk] or null
  float* dq_acc;            // [B*Hq*Sq, 128] fp32, zeroed
  uint16_t *dk, *dv;        // [B*Hkv*Sk, 128] bf16
  unsigned int* status;     // device status word
  int Hq, Hkv, group, Sq, Sk, nbq, nbk;
  int n_tiles;              // key tiles of 128 keys per key/value head
  float scale, scale_log2;
  unsigned long long wait_ns;  // limit of the waits that are not drains (kWaitLimitNs)
  int stall;                // test hook: the MMA warp first waits on a barrier nobody completes
};

namespace bwd {

constexpr int kThreads = 480;
constexpr int kStages = 3;
constexpr int kMaxEntries = 2048;  // (query head, query block) list chunk
constexpr int kDqWarp0 = 8, kTmaWarp = 12, kMmaWarp = 13, kListWarp = 14;
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // one second per wait
constexpr unsigned kErrTimeout = 0x100u;           // | code of the wait that gave up

// shared-memory map (bytes from a 1024-aligned base); every operand tile is stored as
// 64-column (128-byte) halves with the 128-byte swizzle, as TMA writes them
constexpr uint32_t kKVTile = 128 * 128 * 2;  // K or V: [2 d-halves][128 keys][64]
constexpr uint32_t kQTile = 64 * 128 * 2;    // Q or dO of a step: [2 d-halves][64 rows][64]
constexpr uint32_t kOffK = 0;
constexpr uint32_t kOffV = kKVTile;
constexpr uint32_t kOffQ = 2 * kKVTile;                  // [kStages]
constexpr uint32_t kOffDO = kOffQ + kStages * kQTile;    // [kStages]
constexpr uint32_t kDSTile = 128 * 64 * 2;               // dS^T [128 keys][64 queries] bf16
constexpr uint32_t kOffDS = kOffDO + kStages * kQTile;   // dS^T [2] (one per step slot)
constexpr uint32_t kOffRow = kOffDS + 2 * kDSTile;       // [kStages] -lse[64], -D[64]
constexpr uint32_t kOffList = kOffRow + kStages * 512;
constexpr uint32_t kOffCtl = kOffList + kMaxEntries * 4;
constexpr uint32_t kSmemBytes = kOffCtl + 1024 + 1024;  // + alignment slack

constexpr uint32_t kTmemCols = 512;
// two step slots: slot b (steps g with g & 1 == b) holds S^T (then the step's P^T) at
// 128 b and dP^T (then the step's dQ^T) at 128 b + 64
constexpr uint32_t kColSlot = 128, kColDPOff = 64, kColDV = 256, kColDK = 384;

struct Ctl {
  uint64_t kv_full;
  uint64_t ld_full[kStages], ld_empty[kStages];
  // per step slot b (one phase per step of that slot)
  uint64_t s_full[2], dp_full[2];    // S^T (dP^T) of the step is in TMEM
  uint64_t p_full[2], ds_full[2];    // the 8 gradient warps wrote P^T (TMEM) / dS^T (SMEM)
  uint64_t dq_full[2], dq_empty[2];  // dK, dQ^T of the step done (dS^T read) / dQ^T read out
  uint64_t acc_full, acc_full_dk, drain;  // dV (dK) complete; every MMA of warp 13 done
  uint64_t drain_dq;  // every dQ^T MMA of the second issuing thread has completed
  uint64_t never;  // completed by nobody (the timeout test hook waits on it)
  int n_entries, go;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Ctl) <= 1024, "control block too large");
static_assert(kOffDS % 1024 == 0 && kOffQ % 1024 == 0 && kOffDO % 1024 == 0, "swizzle atoms");
static_assert(kSmemBytes <= 227 * 1024, "backward SMEM");

// Bounded wait on an mbarrier phase (as in the forward): gives up after the launch's
// limit a.wait_ns, recording `code` in the status word and raising the abort flag, or as
// soon as another role has raised the flag -- unless `drain`, for copies / MMAs still in
// flight, which always runs to the full kWaitLimitNs.
// (The control block type is a parameter: both backward kernels use these waits.)
template <class CtlT>
__device__ __forceinline__ bool wait(uint64_t* bar, uint32_t parity, CtlT* ctl, const BwdArgs& a,
                                     unsigned code, bool drain = false) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t limit = drain ? kWaitLimitNs : a.wait_ns;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (!drain && *reinterpret_cast<volatile int*>(&ctl->abort_flag)) return false;
    if (global_timer_ns() - t0 > limit) {
      *reinterpret_cast<volatile int*>(&ctl->abort_flag) = 1;
      atomicCAS(a.status, 0u, kErrTimeout | code);
      return false;
    }
  }
}

// The same wait by every lane of a warp that goes on to warp-collective TMEM accesses: the
// warp proceeds only if every lane saw the phase complete, so an abort can never leave
// part of a warp inside a .sync.aligned instruction.
template <class CtlT>
__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity, CtlT* ctl,
                                          const BwdArgs& a, unsigned code) {
  const bool w = wait(bar, parity, ctl, a, code);
  return __all_sync(0xffffffffu, w);
}

__device__ __forceinline__ void red_add_f32(float* addr, float x) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(x) : "memory");
}

// list entry: bits 0-15 query block, bits 16-17 which key block(s) of the tile it selects
// (block 64: bit i = key rows 64 i .. 64 i + 63; block 128: bit 0), bits 20-31 query head
// within the group.  First query row of step `sub` (64 rows a step) of a block of `block`
// rows.
__device__ __forceinline__ long long entry_row0(uint32_t e, int sub, const BwdArgs& a, int b,
                                                int hk, int block) {
  const long long bh = (long long)b * a.Hq + hk * a.group + (int)(e >> 20);
  return bh * a.Sq + (long long)(e & 0xFFFFu) * block + sub * 64;
}

template <int BLOCK>
__global__ void __launch_bounds__(kThreads, 1)
    bsa_bwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tdo,
                   const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                   const BwdArgs a) {
  constexpr int kSubQ = BLOCK / 64;  // 64-row steps per query block
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + kOffCtl);
  uint32_t* list = reinterpret_cast<uint32_t*>(smem + kOffList);
  const int warp = (int)(threadIdx.x >> 5);
  const uint32_t lane = threadIdx.x & 31;

  const int tile = (int)(blockIdx.x % (unsigned)a.n_tiles);   // the CTA's key tile
  const int bkv = (int)(blockIdx.x / (unsigned)a.n_tiles);    // b * Hkv + hk
  const int b = bkv / a.Hkv, hk = bkv - b * a.Hkv;
  // valid keys of the tile's key block(s): vk[i] for key rows 64 i .. (block 64)
  int vk[2] = {0, 0};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int kb = BLOCK == 64 ? 2 * tile + i : tile;
    if ((BLOCK == 64 || i == 0) && kb < a.nbk) {
      const int v = a.vbs != nullptr ? a.vbs[kb] : BLOCK;
      vk[i] = v < 0 ? 0 : (v > BLOCK ? BLOCK : v);
    }
  }

  if (threadIdx.x == 0) {
    mbar_init(&ctl->kv_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ctl->ld_full[s], 1);
      mbar_init(&ctl->ld_empty[s], 2);  // one commit from each MMA-issuing thread
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctl->s_full[i], 1);
      mbar_init(&ctl->dp_full[i], 1);
      mbar_init(&ctl->p_full[i], 8);
      mbar_init(&ctl->ds_full[i], 8);
      mbar_init(&ctl->dq_full[i], 1);
      mbar_init(&ctl->dq_empty[i], 4);
    }
    mbar_init(&ctl->acc_full, 1);
    mbar_init(&ctl->acc_full_dk, 1);
    mbar_init(&ctl->drain, 1);
    mbar_init(&ctl->drain_dq, 1);
    mbar_init(&ctl->never, 1);
    ctl->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kTmaWarp && lane == 0) {
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tdo);
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&ctl->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;  // the warp's TMEM lanes

  uint32_t g = 0;               // steps so far (every role counts alike)
  int scan_h = 0, scan_qb = 0;  // list warp: position in the (head, query block) scan
  bool kv_issued = false;       // TMA warp
  uint32_t fills[kStages] = {0, 0, 0};
  bool ok = true;               // this role has not given up
  while (true) {
    __syncthreads();  // every role is done with the previous chunk's list
    if (warp == kListWarp) {
      // the column of the block map: (query head h of the group, query block qb) pairs
      // that select the key block, ascending, 128 query blocks per round trip
      int cnt = 0;
      while (scan_h < a.group && cnt + 128 <= kMaxEntries) {
        const long long bh = (long long)b * a.Hq + hk * a.group + scan_h;
        uint32_t sel[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int qb = scan_qb + 32 * u + (int)lane;
          sel[u] = 0;
          if (qb < a.nbq) {
            const int8_t* row = a.bitmap + (bh * a.nbq + qb) * (long long)a.nbk;
            if (BLOCK == 128) {
              sel[u] = row[tile] != 0 ? 1u : 0u;
            } else {
              sel[u] = row[2 * tile] != 0 ? 1u : 0u;
              if (2 * tile + 1 < a.nbk && row[2 * tile + 1] != 0) sel[u] |= 2u;
            }
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t ballot = __ballot_sync(0xffffffffu, sel[u] != 0);
          if (sel[u])
            list[cnt + __popc(ballot & ((1u << lane) - 1u))] =
                ((uint32_t)scan_h << 20) | (sel[u] << 16) | (uint32_t)(scan_qb + 32 * u + lane);
          cnt += __popc(ballot);
        }
        scan_qb += 128;
        if (scan_qb >= a.nbq) {
          scan_qb = 0;
          ++scan_h;
        }
      }
      if (lane == 0) {
        ctl->n_entries = cnt;
        ctl->go = (cnt > 0 && *reinterpret_cast<volatile int*>(&ctl->abort_flag) == 0) ? 1 : 0;
      }
    }
    __syncthreads();
    if (!ctl->go) break;
    const int n_steps = ctl->n_entries * kSubQ;
    const uint32_t g0 = g;
    g += (uint32_t)n_steps;
    if (!ok) continue;

    if (warp == kTmaWarp) {
      // ---------------------------------------------------------------- copies
      if (lane == 0) {
        if (!kv_issued) {
          const uint64_t pol = policy_evict_first();
          mbar_arrive_expect_tx(&ctl->kv_full, 2 * kKVTile);
          tma_load_3d_hint(smem + kOffK, &tk, &ctl->kv_full, 0, 128 * tile, bkv, pol);
          tma_load_3d_hint(smem + kOffK + kKVTile / 2, &tk, &ctl->kv_full, 64, 128 * tile, bkv,
                           pol);
          tma_load_3d_hint(smem + kOffV, &tv, &ctl->kv_full, 0, 128 * tile, bkv, pol);
          tma_load_3d_hint(smem + kOffV + kKVTile / 2, &tv, &ctl->kv_full, 64, 128 * tile, bkv,
                           pol);
          kv_issued = true;
        }
        for (int i = 0; i < n_steps; ++i) {
          const uint32_t gg = g0 + i, st = gg % kStages;
          if (gg >= (uint32_t)kStages &&
              !wait(&ctl->ld_empty[st], ((gg / kStages) + 1) & 1, ctl, a, 0x41)) {
            ok = false;
            break;
          }
          const long long row0 = entry_row0(list[i / kSubQ], i % kSubQ, a, b, hk, BLOCK);
          uint8_t* qs = smem + kOffQ + st * kQTile;
          uint8_t* os = smem + kOffDO + st * kQTile;
          float* rs = reinterpret_cast<float*>(smem + kOffRow + st * 512);
          mbar_arrive_expect_tx(&ctl->ld_full[st], 2 * kQTile + 512);
          tma_load_2d(qs, &tq, &ctl->ld_full[st], 0, (int)row0);
          tma_load_2d(qs + kQTile / 2, &tq, &ctl->ld_full[st], 64, (int)row0);
          tma_load_2d(os, &tdo, &ctl->ld_full[st], 0, (int)row0);
          tma_load_2d(os + kQTile / 2, &tdo, &ctl->ld_full[st], 64, (int)row0);
          bulk_load(rs, a.nlse + row0, 256, &ctl->ld_full[st]);
          bulk_load(rs + 64, a.nD + row0, 256, &ctl->ld_full[st]);
          ++fills[st];
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    } else if (warp == kMmaWarp) {
      // ---------------------------------------------------------------- MMA issue
      // the whole warp runs the loop (waits voted), lane 0 alone issues
      {
        constexpr uint32_t kIdescS = idesc_bf16_f32(128, 64, false, false);
        constexpr uint32_t kIdescG = idesc_bf16_f32(128, 128, false, true);
        const uint64_t k_kmaj = smem_desc_sw128(smem_addr(smem + kOffK), 16, 1024);
        const uint64_t v_kmaj = smem_desc_sw128(smem_addr(smem + kOffV), 16, 1024);
        if (g0 == 0 && !wait_warp(&ctl->kv_full, 0, ctl, a, 0x42)) ok = false;
        if (ok && a.stall) {
          // test hook: wait on a barrier no role ever completes, so the wait runs out,
          // the status word records code 0x5f and every role unwinds
          wait_warp(&ctl->never, 0, ctl, a, 0x5f);
          ok = false;
        }
        // S^T (dP^T) of step gg into its slot: A = K (V) K-major, B = Q (dO) K-major,
        // K = d in 8 steps
        auto issue_sd = [&](uint32_t gg, bool dp) {
          const uint32_t st = gg % kStages, b = gg & 1;
          const uint64_t ad = dp ? v_kmaj : k_kmaj;
          const uint64_t bd =
              smem_desc_sw128(smem_addr(smem + (dp ? kOffDO : kOffQ) + st * kQTile), 16, 1024);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint64_t oa = ((k >> 2) * (kKVTile / 2) + (k & 3) * 32) >> 4;
            const uint64_t ob = ((k >> 2) * (kQTile / 2) + (k & 3) * 32) >> 4;
            warp_mma_ss(tmem + kColSlot * b + (dp ? kColDPOff : 0u), ad + oa, bd + ob, kIdescS,
                        k > 0 ? 1u : 0u);
          }
          warp_mma_commit(dp ? &ctl->dp_full[b] : &ctl->s_full[b]);
        };
        // the step's Q, dO have landed
        auto landed = [&](uint32_t gg) {
          return wait_warp(&ctl->ld_full[gg % kStages], (gg / kStages) & 1, ctl, a, 0x43);
        };
        // dP^T of step gg overwrites the slot's dQ^T of step gg - 2: read out by then
        auto dq_read = [&](uint32_t gg) {
          return gg < 2 || wait_warp(&ctl->dq_empty[gg & 1], ((gg - 2) >> 1) & 1, ctl, a, 0x47);
        };
        if (ok) {
          if (!landed(g0) || !dq_read(g0)) {
            ok = false;
          } else {
            tc_fence_after();
            issue_sd(g0, false);
            issue_sd(g0, true);
          }
        }
        for (int i = 0; i < n_steps && ok; ++i) {
          const uint32_t gg = g0 + i, st = gg % kStages, b = gg & 1;
          // S^T of the next step into the other slot, ahead of this step's dV: that slot's
          // previous P^T (step gg - 1) was read by dV issued earlier on this thread
          if (i + 1 < n_steps) {
            if (!landed(gg + 1)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_sd(gg + 1, false);
          }
          // dV += P^T dO: A = P^T (TMEM, 64 query columns as 32 packed), B = dO MN-major
          if (!wait_warp(&ctl->p_full[b], (gg >> 1) & 1, ctl, a, 0x44)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t do_mn =
              smem_desc_sw128(smem_addr(smem + kOffDO + st * kQTile), kQTile / 2, 1024);
          const uint32_t tS = tmem + kColSlot * b;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            warp_mma_ts(tmem + kColDV, tS + 32 * (kk >> 1) + 8 * (kk & 1),
                        do_mn + ((kk * 2048) >> 4), kIdescG, (gg > 0 || kk > 0) ? 1u : 0u);
          warp_mma_commit(&ctl->ld_empty[st]);  // this thread's readers of the stage are done
          // dP^T of the next step into the other slot once its dQ^T (step gg - 1) is out
          if (i + 1 < n_steps) {
            if (!dq_read(gg + 1)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_sd(gg + 1, true);
          }
        }
      }
    } else if (warp == kListWarp) {
      // ---------------------------------------------------------------- dK, dQ issue
      // The two contractions that take dS^T, on a second issuing thread: they depend on no
      // other MMA of the step (dS^T comes from SMEM), and one thread alone cannot issue a
      // step's 32 MMAs as fast as the tensor pipe runs them.
      //   dK  += dS^T Q    (A = dS^T K-major, B = Q MN-major, K = queries in 4 steps)
      //   dQ^T = K^T dS^T  (both MN-major, K = keys in 8 steps) over the step slot's dP^T
      // (the whole warp runs the loop, lane 0 alone issues)
      {
        constexpr uint32_t kIdescG = idesc_bf16_f32(128, 128, false, true);
        constexpr uint32_t kIdescQ = idesc_bf16_f32(128, 64, true, true);
        const uint64_t k_mn = smem_desc_sw128(smem_addr(smem + kOffK), kKVTile / 2, 1024);
        if (g0 == 0 && !wait_warp(&ctl->kv_full, 0, ctl, a, 0x51)) ok = false;
        for (int i = 0; i < n_steps && ok; ++i) {
          const uint32_t gg = g0 + i, db = gg & 1, st = gg % kStages;
          const uint64_t ds_mn = smem_desc_sw128(smem_addr(smem + kOffDS + db * kDSTile), 8192, 1024);
          const uint64_t ds_kmaj = smem_desc_sw128(smem_addr(smem + kOffDS + db * kDSTile), 16, 1024);
          if (!wait_warp(&ctl->ds_full[db], (gg >> 1) & 1, ctl, a, 0x52)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t q_mn =
              smem_desc_sw128(smem_addr(smem + kOffQ + st * kQTile), kQTile / 2, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            warp_mma_ss(tmem + kColDK, ds_kmaj + ((kk * 32) >> 4), q_mn + ((kk * 2048) >> 4),
                        kIdescG, (gg > 0 || kk > 0) ? 1u : 0u);
          warp_mma_commit(&ctl->ld_empty[st]);  // this thread's readers of the stage are done
          // dQ^T over the slot's dP^T, which the gradient warps have read (dS^T is ready)
#pragma unroll
          for (int k = 0; k < 8; ++k)
            warp_mma_ss(tmem + kColSlot * db + kColDPOff, k_mn + ((k * 2048) >> 4),
                        ds_mn + ((k * 2048) >> 4), kIdescQ, k > 0 ? 1u : 0u);
          warp_mma_commit(&ctl->dq_full[db]);
        }
      }
    } else if (warp < 8) {
      // ---------------------------------------------------------------- P^T and dS^T
      const int wg = warp >> 2;
      const int r = (warp & 3) * 32 + (int)lane;  // key row of the tile
      const int kbi = BLOCK == 64 ? (r >> 6) : 0;
      const bool key_ok = (r & (BLOCK - 1)) < (kbi ? vk[1] : vk[0]);
      for (int i = 0; i < n_steps; ++i) {
        const uint32_t gg = g0 + i, st = gg % kStages, b = gg & 1;
        // block 64: this half of the tile is key block kbi, which the entry may not select
        const bool valid = BLOCK == 128 ? key_ok
                                        : key_ok && ((list[i / kSubQ] >> (16 + kbi)) & 1u);
        const uint32_t tS = tmem + lane_base + kColSlot * b + 32 * wg, tDP = tS + kColDPOff;
        uint8_t* ds_row = smem + kOffDS + b * kDSTile + (r >> 3) * 1024 + (r & 7) * 128;
        const float* nlse_s = reinterpret_cast<const float*>(smem + kOffRow + st * 512) + 32 * wg;
        const float* nD_s = nlse_s + 64;
        // -lse and -D of the step have landed (the stage is not refilled before dK of this
        // step, which waits for this warp); -lse is read into registers while S^T is still
        // being computed
        if (!wait_warp(&ctl->ld_full[st], (gg / kStages) & 1, ctl, a, 0x48)) {
          ok = false;
          break;
        }
        float4 l4[8];
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) l4[c4] = reinterpret_cast<const float4*>(nlse_s)[c4];
        if (!wait_warp(&ctl->s_full[b], (gg >> 1) & 1, ctl, a, 0x49)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[32];
        tmem_ld_32x32b_x32(tS, sr);
        tmem_wait_ld();
        // p = 2^(s scale log2(e) - lse): pairs of columns per fp32x2 instruction; a key the
        // query block did not select gives 0, and so does a row with no attended key
        // (its -lse is -inf)
        float p[32];
        if (valid) {
          const uint64_t c2 = f32x2(a.scale_log2, a.scale_log2);
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            const int c = 4 * c4;
            const uint64_t x01 = fma_f32x2(f32x2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])),
                                           c2, f32x2(l4[c4].x, l4[c4].y));
            const uint64_t x23 = fma_f32x2(
                f32x2(__uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3])), c2,
                f32x2(l4[c4].z, l4[c4].w));
            float x[4];
            split_f32x2(x01, x[0], x[1]);
            split_f32x2(x23, x[2], x[3]);
#pragma unroll
            for (int j = 0; j < 4; ++j) p[c + j] = fast_exp2(x[j]);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) p[c] = 0.0f;
        }
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(p[2 * j], p[2 * j + 1]);
        tmem_st_32x32b_x16(tS, pk);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->p_full[b]);
        float4 d4[8];  // -D, read while dP^T is still being computed
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) d4[c4] = reinterpret_cast<const float4*>(nD_s)[c4];
        if (!wait_warp(&ctl->dp_full[b], (gg >> 1) & 1, ctl, a, 0x4a)) {
          ok = false;
          break;
        }
        tc_fence_after();
        tmem_ld_32x32b_x32(tDP, sr);
        tmem_wait_ld();
        if (valid) {  // dS = p (dP - D), without the factor scale
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            const int c = 4 * c4;
            const uint64_t t01 = add_f32x2(f32x2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])),
                                           f32x2(d4[c4].x, d4[c4].y));
            const uint64_t t23 = add_f32x2(
                f32x2(__uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3])),
                f32x2(d4[c4].z, d4[c4].w));
            split_f32x2(mul_f32x2(f32x2(p[c], p[c + 1]), t01), p[c], p[c + 1]);
            split_f32x2(mul_f32x2(f32x2(p[c + 2], p[c + 3]), t23), p[c + 2], p[c + 3]);
          }
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(p[2 * j], p[2 * j + 1]);
        // the slot's SMEM dS^T tile is free once dK and dQ^T of step gg - 2 have read it
        if (gg >= 2 && !wait_warp(&ctl->dq_full[b], ((gg - 2) >> 1) & 1, ctl, a, 0x50)) {
          ok = false;
          break;
        }
        // dS^T row r, query columns 32 wg .. 32 wg + 31: 16-byte chunks 4 wg .. 4 wg + 3
        // of the 128-byte row, placed by the 128-byte swizzle (chunk ^ row % 8)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int phys = (4 * wg + c) ^ (r & 7);
          *reinterpret_cast<uint4*>(ds_row + phys * 16) =
              make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->ds_full[b]);
      }
    } else if (warp >= kDqWarp0 && warp < kDqWarp0 + 4) {
      // ---------------------------------------------------------------- dQ reductions
      const int d = (warp & 3) * 32 + (int)lane;  // d column (TMEM lane of dQ^T)
      for (int i = 0; i < n_steps; ++i) {
        const uint32_t gg = g0 + i, db = gg & 1;
        const long long row0 = entry_row0(list[i / kSubQ], i % kSubQ, a, b, hk, BLOCK);
        if (!wait_warp(&ctl->dq_full[db], (gg >> 1) & 1, ctl, a, 0x4b)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t v0[32], v1[32];
        tmem_ld_32x32b_x32(tmem + lane_base + kColSlot * db + kColDPOff, v0);
        tmem_ld_32x32b_x32(tmem + lane_base + kColSlot * db + kColDPOff + 32, v1);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->dq_empty[db]);
        float* dst = a.dq_acc + row0 * 128 + d;
#pragma unroll
        for (int q = 0; q < 32; ++q) red_add_f32(dst + q * 128, __uint_as_float(v0[q]));
#pragma unroll
        for (int q = 0; q < 32; ++q) red_add_f32(dst + (32 + q) * 128, __uint_as_float(v1[q]));
      }
    }
  }

  // ------------------------------------------------------------------ dK, dV epilogue
  // (dK takes the factor scale that dS^T left out)
  const bool any = g > 0;
  if (warp == kMmaWarp) {
    if (any && ok) warp_mma_commit(&ctl->acc_full);
    // every MMA issued has completed before TMEM can be released
    warp_mma_commit(&ctl->drain);
    wait(&ctl->drain, 0, ctl, a, 0x4c, true);
    __syncwarp();
  } else if (warp == kListWarp) {
    // every MMA this warp issued has completed before TMEM goes
    if (any && ok) warp_mma_commit(&ctl->acc_full_dk);
    warp_mma_commit(&ctl->drain_dq);
    wait(&ctl->drain_dq, 0, ctl, a, 0x53, true);
    __syncwarp();
  } else if (warp == kTmaWarp) {
    if (lane == 0) {  // every copy issued has landed before the CTA exits
      if (kv_issued) wait(&ctl->kv_full, 0, ctl, a, 0x4d, true);
      for (int s = 0; s < kStages; ++s)
        if (fills[s]) wait(&ctl->ld_full[s], (fills[s] - 1) & 1, ctl, a, 0x4e, true);
    }
    __syncwarp();
  } else if (warp < 8) {
    const int r = (warp & 3) * 32 + (int)lane;
    const bool is_dk = warp >= 4;
    const bool row_ok = BLOCK == 128 || 128 * tile + r < a.Sk;  // a lone last block-64 key block
    const float sc = is_dk ? a.scale : 1.0f;
    uint16_t* dst = (is_dk ? a.dk : a.dv) + ((long long)bkv * a.Sk + 128 * tile + r) * 128;
    bool have = false;
    if (any && ok) {
      have = wait_warp(is_dk ? &ctl->acc_full_dk : &ctl->acc_full, 0, ctl, a, 0x4f);
      tc_fence_after();
    }
    if (have || !any) {
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        if (have) {
          tmem_ld_32x32b_x32(tmem + lane_base + (is_dk ? kColDK : kColDV) + 32 * c, v);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = 0u;  // no query row attends this block
        }
        if (row_ok) {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            reinterpret_cast<uint4*>(dst + 32 * c)[j] = make_uint4(
                pack_bf16x2(__uint_as_float(v[8 * j]) * sc, __uint_as_float(v[8 * j + 1]) * sc),
                pack_bf16x2(__uint_as_float(v[8 * j + 2]) * sc, __uint_as_float(v[8 * j + 3]) * sc),
                pack_bf16x2(__uint_as_float(v[8 * j + 4]) * sc, __uint_as_float(v[8 * j + 5]) * sc),
                pack_bf16x2(__uint_as_float(v[8 * j + 6]) * sc, __uint_as_float(v[8 * j + 7]) * sc));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace bwd
}  // namespace vsa
