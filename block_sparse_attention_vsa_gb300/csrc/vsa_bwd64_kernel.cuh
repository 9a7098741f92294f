// vsa_bwd64_kernel.cuh -- backward of the block-sparse attention forward for block 64, one
// CTA per 64-key block, query rows on the MMA M dimension.
//
// What it computes: the same gradients as vsa_bwd_kernel.cuh ("FastVideo
// block_sparse_attn_sm100a.py", module docstring: the backward consumes the forward's base-2
// lse), p_ij = 2^(s_ij scale log2 e - lse_i), ds_ij = p_ij (dout_i . v_j - D_i),
// dq_i = scale sum_j ds_ij k_j, dk_j = scale sum_i ds_ij q_i, dv_j = sum_i p_ij dout_i.
//
// Why a kernel of its own: the block-128 kernel (vsa_bwd_kernel.cuh) puts the keys of one
// block on the MMA M dimension (M = 128).  With 64-key blocks that layout needs a pair of
// key blocks per CTA walking the union of the query blocks selecting either, so keys of
// the block a query block did not select are computed and masked (43 % of the MMA work on
// a 25 %-dense random selection).  Here a CTA owns ONE key block and puts query rows on
// M: a step takes two consecutive entries of the block-map column (two query blocks that
// both select this key block, 128 rows), so no MMA work is masked except the second half
// of a chunk's odd last step.  The per-row -lse and -D are then one value per thread.
//
// bsa_bwd64_kernel, one CTA per (batch, key/value head, key block), per step t (128 query
// rows, the entries 2i and 2i + 1 of the list chunk; slot b = t & 1):
//   S    = Q K^T     (M = 128 rows, N = 64 keys, K = d)     -> TMEM slot b, columns 0-63
//   dP   = dO V^T                                          -> TMEM slot b, columns 64-127
//   P, dS formed by the gradient warps (thread = query row) and written to SMEM as bf16
//   [128 rows][64 keys] tiles (dS without the factor scale)
//   dV^T += dO^T P   (M = 128 d, N = 64 keys, K = 128 rows; both operands MN-major)
//   dK^T += Q^T dS
//   dQ^T  = K^T dS^T (M = 128 d, N = 128 rows, K = 64 keys; A MN-major, B = dS K-major)
// and the dQ warps add dQ^T into the fp32 accumulator with coalesced reductions (thread =
// d column).  dV^T and dK^T stay in TMEM for the whole key block; the epilogue writes dv
// and dk (dk times scale) as bf16.
//
// Roles (15 warps):
//   warps 0-7   gradient warps: warp w handles rows 32 (w % 4) .. + 31 (its TMEM lane
//               quarter) and keys 32 (w / 4) .. + 31; after the last step warps 0-3 store
//               dv and warps 4-7 dk.
//   warps 8-11  dQ warps: thread = d column (TMEM lane of dQ^T).
//   warp 12     TMA: K, V once; per step Q, dO (two 64-row boxes per d-half) and -lse, -D
//               into a 2-stage ring.
//   warp 13     MMA issuer of S, dP (one step ahead) and dQ^T; owns the TMEM allocation.
//   warp 14     list: compacts the block-map column into the entry list (in chunks);
//               during the steps it issues dV^T and dK^T.
// Both issuing warps run their loops converged; the lane elect.sync picks issues.
// TMEM (512 columns): step slots at 0 and 128 (S, then dP), dQ^T 256-383, dV^T 384-447,
// dK^T 448-511.
// Ordering: S/dP of step t + 1 are issued once the slot's previous reader (the gradient
// warps, step t - 1) is done; P_t (dS_t) overwrites the SMEM tile once dV^T_{t-1}
// (dK^T_{t-1} and dQ^T_{t-1}) completed; dQ^T_t waits until the dQ warps have read dQ^T
// of step t - 1.  A Q/dO stage is free once S, dP (first issuer) and dV^T, dK^T (second)
// of its step completed.  Every mbarrier wait is bounded as in the other kernels.
#pragma once

#include <cuda.h>

#include <cstdint>

#include "sm103_ptx.cuh"
#include "vsa_bwd_kernel.cuh"

namespace vsa {
namespace bwd64 {

constexpr int kThreads = 480;
constexpr int kStages = 2;
constexpr int kMaxEntries = 2048;  // (query head, query block) list chunk
constexpr int kDqWarp0 = 8, kTmaWarp = 12, kMmaWarp = 13, kListWarp = 14;

// shared-memory map (bytes from a 1024-aligned base); operand tiles are 64-column
// (128-byte) halves with the 128-byte swizzle, as TMA writes them
constexpr uint32_t kKVTile = 64 * 128 * 2;    // K or V: [2 d-halves][64 keys][64]
constexpr uint32_t kQTile = 128 * 128 * 2;    // Q or dO of a step: [2 d-halves][128 rows][64]
constexpr uint32_t kPTile = 128 * 64 * 2;     // P or dS: [128 rows][64 keys]
constexpr uint32_t kOffK = 0;
constexpr uint32_t kOffV = kKVTile;
constexpr uint32_t kOffQ = 2 * kKVTile;                  // [kStages]
constexpr uint32_t kOffDO = kOffQ + kStages * kQTile;    // [kStages]
constexpr uint32_t kOffP = kOffDO + kStages * kQTile;
constexpr uint32_t kOffDS = kOffP + kPTile;
constexpr uint32_t kOffRow = kOffDS + kPTile;            // [kStages] -lse[128], -D[128]
constexpr uint32_t kOffList = kOffRow + kStages * 1024;
constexpr uint32_t kOffCtl = kOffList + kMaxEntries * 4;
constexpr uint32_t kSmemBytes = kOffCtl + 1024 + 1024;  // + alignment slack

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColSlot = 128, kColDPOff = 64, kColDQ = 256, kColDV = 384, kColDK = 448;

struct Ctl {
  uint64_t kv_full;
  uint64_t ld_full[kStages], ld_empty[kStages];
  uint64_t s_full[2], dp_full[2];  // S (dP) of the slot's step is in TMEM
  uint64_t slot_free[2];           // the 8 gradient warps have read S and dP of the slot
  uint64_t p_full, ds_full;        // the 8 gradient warps wrote P (dS) of the step to SMEM
  uint64_t p_free;                 // dV^T of the step completed: the P tile is free
  uint64_t ds_free;                // dK^T and dQ^T of the step completed: the dS tile is free
  uint64_t dq_full, dq_empty;      // dQ^T of the step is in TMEM / has been read out
  uint64_t acc_full;               // every dV^T, dK^T MMA completed
  uint64_t drain, drain2;          // every MMA of the first (second) issuer completed
  uint64_t never;                  // completed by nobody (the timeout test hook waits on it)
  int n_entries, go;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Ctl) <= 1024, "control block too large");
static_assert(kOffQ % 1024 == 0 && kOffDO % 1024 == 0 && kOffP % 1024 == 0 &&
                  kOffDS % 1024 == 0 && kOffRow % 16 == 0,
              "swizzle atoms, bulk copies");
static_assert(kSmemBytes <= 227 * 1024, "backward SMEM");
static_assert(kMaxEntries % 2 == 0, "a step takes two entries");

using bwd::wait;
using bwd::wait_warp;

__global__ void __launch_bounds__(kThreads, 1)
    bsa_bwd64_kernel(const __grid_constant__ CUtensorMap tq,
                     const __grid_constant__ CUtensorMap tdo,
                     const __grid_constant__ CUtensorMap tk,
                     const __grid_constant__ CUtensorMap tv, const BwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + kOffCtl);
  uint32_t* list = reinterpret_cast<uint32_t*>(smem + kOffList);
  const int warp = (int)(threadIdx.x >> 5);
  const uint32_t lane = threadIdx.x & 31;

  const int kb = (int)(blockIdx.x % (unsigned)a.nbk);      // the CTA's key block
  const int bkv = (int)(blockIdx.x / (unsigned)a.nbk);     // b * Hkv + hk
  const int b = bkv / a.Hkv, hk = bkv - b * a.Hkv;
  int vk = 64;  // valid keys of the block
  if (a.vbs != nullptr) {
    const int v = a.vbs[kb];
    vk = v < 0 ? 0 : (v > 64 ? 64 : v);
  }

  if (threadIdx.x == 0) {
    mbar_init(&ctl->kv_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ctl->ld_full[s], 1);
      mbar_init(&ctl->ld_empty[s], 2);  // one commit from each issuing warp
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctl->s_full[i], 1);
      mbar_init(&ctl->dp_full[i], 1);
      mbar_init(&ctl->slot_free[i], 8);
    }
    mbar_init(&ctl->p_full, 8);
    mbar_init(&ctl->ds_full, 8);
    mbar_init(&ctl->p_free, 1);
    mbar_init(&ctl->ds_free, 2);  // dK^T (second issuer) and dQ^T (first)
    mbar_init(&ctl->dq_full, 1);
    mbar_init(&ctl->dq_empty, 4);
    mbar_init(&ctl->acc_full, 1);
    mbar_init(&ctl->drain, 1);
    mbar_init(&ctl->drain2, 1);
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
  uint32_t fills0 = 0, fills1 = 0;
  bool ok = true;               // this role has not given up
  while (true) {
    __syncthreads();  // every role is done with the previous chunk's list
    if (warp == kListWarp) {
      // the column kb of the block map: (query head h of the group, query block qb) pairs
      // that select the key block, ascending, 128 query blocks per round trip
      int cnt = 0;
      while (scan_h < a.group && cnt + 128 <= kMaxEntries) {
        const long long bh = (long long)b * a.Hq + hk * a.group + scan_h;
        bool sel[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int qb = scan_qb + 32 * u + (int)lane;
          sel[u] = qb < a.nbq && a.bitmap[(bh * a.nbq + qb) * (long long)a.nbk + kb] != 0;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t ballot = __ballot_sync(0xffffffffu, sel[u]);
          if (sel[u])
            list[cnt + __popc(ballot & ((1u << lane) - 1u))] =
                ((uint32_t)scan_h << 20) | (uint32_t)(scan_qb + 32 * u + lane);
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
    const int n_entries = ctl->n_entries;
    const int n_steps = (n_entries + 1) / 2;
    const uint32_t g0 = g;
    g += (uint32_t)n_steps;
    if (!ok) continue;

    if (warp == kTmaWarp) {
      // ---------------------------------------------------------------- copies
      if (lane == 0) {
        if (!kv_issued) {
          const uint64_t pol = policy_evict_first();
          mbar_arrive_expect_tx(&ctl->kv_full, 2 * kKVTile);
          tma_load_3d_hint(smem + kOffK, &tk, &ctl->kv_full, 0, 64 * kb, bkv, pol);
          tma_load_3d_hint(smem + kOffK + kKVTile / 2, &tk, &ctl->kv_full, 64, 64 * kb, bkv,
                           pol);
          tma_load_3d_hint(smem + kOffV, &tv, &ctl->kv_full, 0, 64 * kb, bkv, pol);
          tma_load_3d_hint(smem + kOffV + kKVTile / 2, &tv, &ctl->kv_full, 64, 64 * kb, bkv,
                           pol);
          kv_issued = true;
        }
        for (int i = 0; i < n_steps; ++i) {
          const uint32_t gg = g0 + i, st = gg % kStages;
          if (gg >= (uint32_t)kStages &&
              !wait(&ctl->ld_empty[st], ((gg / kStages) + 1) & 1, ctl, a, 0x61)) {
            ok = false;
            break;
          }
          // rows 0-63 from entry 2i, rows 64-127 from entry 2i + 1; an odd chunk's last
          // step loads entry 2i twice (its second half is masked, but stays finite)
          const uint32_t e0 = list[2 * i];
          const uint32_t e1 = 2 * i + 1 < n_entries ? list[2 * i + 1] : e0;
          const long long r0 = bwd::entry_row0(e0, 0, a, b, hk, 64);
          const long long r1 = bwd::entry_row0(e1, 0, a, b, hk, 64);
          uint8_t* qs = smem + kOffQ + st * kQTile;
          uint8_t* os = smem + kOffDO + st * kQTile;
          float* rs = reinterpret_cast<float*>(smem + kOffRow + st * 1024);
          uint64_t* bar = &ctl->ld_full[st];
          mbar_arrive_expect_tx(bar, 2 * kQTile + 1024);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            tma_load_2d(qs + h * (kQTile / 2), &tq, bar, 64 * h, (int)r0);
            tma_load_2d(qs + h * (kQTile / 2) + kQTile / 4, &tq, bar, 64 * h, (int)r1);
            tma_load_2d(os + h * (kQTile / 2), &tdo, bar, 64 * h, (int)r0);
            tma_load_2d(os + h * (kQTile / 2) + kQTile / 4, &tdo, bar, 64 * h, (int)r1);
          }
          bulk_load(rs, a.nlse + r0, 256, bar);
          bulk_load(rs + 64, a.nlse + r1, 256, bar);
          bulk_load(rs + 128, a.nD + r0, 256, bar);
          bulk_load(rs + 192, a.nD + r1, 256, bar);
          if (st) ++fills1; else ++fills0;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    } else if (warp == kMmaWarp) {
      // ---------------------------------------------------------------- S, dP, dQ^T issue
      constexpr uint32_t kIdescS = idesc_bf16_f32(128, 64, false, false);
      constexpr uint32_t kIdescQ = idesc_bf16_f32(128, 128, true, false);
      const uint64_t k_kmaj = smem_desc_sw128(smem_addr(smem + kOffK), 16, 1024);
      const uint64_t v_kmaj = smem_desc_sw128(smem_addr(smem + kOffV), 16, 1024);
      const uint64_t k_mn = smem_desc_sw128(smem_addr(smem + kOffK), kKVTile / 2, 1024);
      const uint64_t ds_kmaj = smem_desc_sw128(smem_addr(smem + kOffDS), 16, 1024);
      if (g0 == 0 && !wait_warp(&ctl->kv_full, 0, ctl, a, 0x62)) ok = false;
      if (ok && a.stall) {
        // test hook: wait on a barrier no role ever completes, so the wait runs out,
        // the status word records code 0x6f and every role unwinds
        wait_warp(&ctl->never, 0, ctl, a, 0x6f);
        ok = false;
      }
      // S and dP of step gg into slot gg & 1 once its copies landed and the gradient warps
      // read the slot's step gg - 2; A = Q (dO) K-major, B = K (V) K-major, K = d in 8 steps
      auto issue_sd = [&](uint32_t gg) -> bool {
        const uint32_t st = gg % kStages, sb = gg & 1;
        if (!wait_warp(&ctl->ld_full[st], (gg / kStages) & 1, ctl, a, 0x63)) return false;
        if (gg >= 2 && !wait_warp(&ctl->slot_free[sb], ((gg - 2) >> 1) & 1, ctl, a, 0x64))
          return false;
        tc_fence_after();
        const uint64_t qd = smem_desc_sw128(smem_addr(smem + kOffQ + st * kQTile), 16, 1024);
        const uint64_t od = smem_desc_sw128(smem_addr(smem + kOffDO + st * kQTile), 16, 1024);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t oa = ((k >> 2) * (kQTile / 2) + (k & 3) * 32) >> 4;
          const uint64_t ob = ((k >> 2) * (kKVTile / 2) + (k & 3) * 32) >> 4;
          warp_mma_ss(tmem + kColSlot * sb, qd + oa, k_kmaj + ob, kIdescS, k > 0 ? 1u : 0u);
        }
        warp_mma_commit(&ctl->s_full[sb]);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t oa = ((k >> 2) * (kQTile / 2) + (k & 3) * 32) >> 4;
          const uint64_t ob = ((k >> 2) * (kKVTile / 2) + (k & 3) * 32) >> 4;
          warp_mma_ss(tmem + kColSlot * sb + kColDPOff, od + oa, v_kmaj + ob, kIdescS,
                      k > 0 ? 1u : 0u);
        }
        warp_mma_commit(&ctl->dp_full[sb]);
        warp_mma_commit(&ctl->ld_empty[st]);  // this warp's readers of the stage are done
        return true;
      };
      if (ok && n_steps > 0 && !issue_sd(g0)) ok = false;
      for (int i = 0; i < n_steps && ok; ++i) {
        const uint32_t gg = g0 + i;
        if (i + 1 < n_steps && !issue_sd(gg + 1)) {
          ok = false;
          break;
        }
        // dQ^T = K^T dS^T: A = K MN-major, B = dS K-major, K = keys in 4 steps; once dS of
        // the step is in SMEM and the dQ warps have read dQ^T of step gg - 1
        if (!wait_warp(&ctl->ds_full, gg & 1, ctl, a, 0x65) ||
            (gg >= 1 && !wait_warp(&ctl->dq_empty, (gg - 1) & 1, ctl, a, 0x66))) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 4; ++k)
          warp_mma_ss(tmem + kColDQ, k_mn + ((k * 2048) >> 4), ds_kmaj + ((k * 32) >> 4),
                      kIdescQ, k > 0 ? 1u : 0u);
        warp_mma_commit(&ctl->dq_full);
        warp_mma_commit(&ctl->ds_free);
      }
    } else if (warp == kListWarp) {
      // ---------------------------------------------------------------- dV^T, dK^T issue
      //   dV^T += dO^T P   (A = dO MN-major, B = P MN-major, K = rows in 8 steps)
      //   dK^T += Q^T dS
      constexpr uint32_t kIdescG = idesc_bf16_f32(128, 64, true, true);
      const uint64_t p_mn = smem_desc_sw128(smem_addr(smem + kOffP), 8192, 1024);
      const uint64_t ds_mn = smem_desc_sw128(smem_addr(smem + kOffDS), 8192, 1024);
      for (int i = 0; i < n_steps && ok; ++i) {
        const uint32_t gg = g0 + i, st = gg % kStages;
        const uint64_t do_mn =
            smem_desc_sw128(smem_addr(smem + kOffDO + st * kQTile), kQTile / 2, 1024);
        const uint64_t q_mn =
            smem_desc_sw128(smem_addr(smem + kOffQ + st * kQTile), kQTile / 2, 1024);
        if (!wait_warp(&ctl->p_full, gg & 1, ctl, a, 0x67)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          warp_mma_ss(tmem + kColDV, do_mn + ((k * 2048) >> 4), p_mn + ((k * 2048) >> 4),
                      kIdescG, (gg > 0 || k > 0) ? 1u : 0u);
        warp_mma_commit(&ctl->p_free);
        if (!wait_warp(&ctl->ds_full, gg & 1, ctl, a, 0x68)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          warp_mma_ss(tmem + kColDK, q_mn + ((k * 2048) >> 4), ds_mn + ((k * 2048) >> 4),
                      kIdescG, (gg > 0 || k > 0) ? 1u : 0u);
        warp_mma_commit(&ctl->ds_free);
        warp_mma_commit(&ctl->ld_empty[st]);  // this warp's readers of the stage are done
      }
    } else if (warp < 8) {
      // ---------------------------------------------------------------- P and dS
      const int wg = warp >> 2;
      const int r = (warp & 3) * 32 + (int)lane;  // query row of the step
      const int ncols = vk - 32 * wg;             // valid keys among this warp's 32
      // P / dS row r, keys 32 wg .. 32 wg + 31: 16-byte chunks 4 wg .. 4 wg + 3 of the
      // 128-byte row, placed by the 128-byte swizzle (chunk ^ row % 8)
      uint8_t* p_row = smem + kOffP + r * 128;
      uint8_t* ds_row = smem + kOffDS + r * 128;
      for (int i = 0; i < n_steps; ++i) {
        const uint32_t gg = g0 + i, st = gg % kStages, sb = gg & 1;
        const uint32_t tS = tmem + lane_base + kColSlot * sb + 32 * wg, tDP = tS + kColDPOff;
        // the row is real unless it is the second half of an odd chunk's last step
        const bool row_ok = r < 64 || 2 * i + 1 < n_entries;
        const float* rs = reinterpret_cast<const float*>(smem + kOffRow + st * 1024);
        if (!wait_warp(&ctl->ld_full[st], (gg / kStages) & 1, ctl, a, 0x69)) {
          ok = false;
          break;
        }
        const float nl = rs[r], nd = rs[128 + r];  // -lse, -D of the row
        if (!wait_warp(&ctl->s_full[sb], (gg >> 1) & 1, ctl, a, 0x6a)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[32];
        tmem_ld_32x32b_x32(tS, sr);
        tmem_wait_ld();
        // p = 2^(s scale log2(e) - lse), pairs of keys per fp32x2 instruction (-lse is -inf
        // for a row with no attended key); masked tail keys and padding rows give 0
        float p[32];
        if (row_ok && ncols > 0) {
          const uint64_t c2 = f32x2(a.scale_log2, a.scale_log2), nl2 = f32x2(nl, nl);
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            float x0, x1;
            split_f32x2(fma_f32x2(f32x2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), c2,
                                  nl2),
                        x0, x1);
            p[c] = fast_exp2(x0);
            p[c + 1] = fast_exp2(x1);
          }
          if (ncols < 32) {
#pragma unroll
            for (int c = 0; c < 32; ++c)
              if (c >= ncols) p[c] = 0.0f;
          }
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) p[c] = 0.0f;
        }
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(p[2 * j], p[2 * j + 1]);
        // the P tile is free once dV^T of the previous step completed
        if (gg >= 1 && !wait_warp(&ctl->p_free, (gg - 1) & 1, ctl, a, 0x6b)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int phys = (4 * wg + c) ^ (r & 7);
          *reinterpret_cast<uint4*>(p_row + phys * 16) =
              make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->p_full);
        if (!wait_warp(&ctl->dp_full[sb], (gg >> 1) & 1, ctl, a, 0x6c)) {
          ok = false;
          break;
        }
        tc_fence_after();
        tmem_ld_32x32b_x32(tDP, sr);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->slot_free[sb]);  // S and dP of the slot are read
        // dS = p (dP - D), without the factor scale
        const uint64_t nd2 = f32x2(nd, nd);
#pragma unroll
        for (int c = 0; c < 32; c += 2)
          split_f32x2(
              mul_f32x2(f32x2(p[c], p[c + 1]),
                        add_f32x2(f32x2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), nd2)),
              p[c], p[c + 1]);
#pragma unroll
        for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(p[2 * j], p[2 * j + 1]);
        // the dS tile is free once dK^T and dQ^T of the previous step completed
        if (gg >= 1 && !wait_warp(&ctl->ds_free, (gg - 1) & 1, ctl, a, 0x6d)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int phys = (4 * wg + c) ^ (r & 7);
          *reinterpret_cast<uint4*>(ds_row + phys * 16) =
              make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->ds_full);
      }
    } else if (warp >= kDqWarp0 && warp < kDqWarp0 + 4) {
      // ---------------------------------------------------------------- dQ reductions
      const int d = (warp & 3) * 32 + (int)lane;  // d column (TMEM lane of dQ^T)
      for (int i = 0; i < n_steps; ++i) {
        const uint32_t gg = g0 + i;
        const long long r0 = bwd::entry_row0(list[2 * i], 0, a, b, hk, 64);
        const bool second = 2 * i + 1 < n_entries;
        const long long r1 = second ? bwd::entry_row0(list[2 * i + 1], 0, a, b, hk, 64) : r0;
        if (!wait_warp(&ctl->dq_full, gg & 1, ctl, a, 0x6e)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t v0[32], v1[32];
        tmem_ld_32x32b_x32(tmem + lane_base + kColDQ, v0);
        tmem_ld_32x32b_x32(tmem + lane_base + kColDQ + 32, v1);
        tmem_wait_ld();
        float* dst = a.dq_acc + r0 * 128 + d;
#pragma unroll
        for (int q = 0; q < 32; ++q) bwd::red_add_f32(dst + q * 128, __uint_as_float(v0[q]));
#pragma unroll
        for (int q = 0; q < 32; ++q)
          bwd::red_add_f32(dst + (32 + q) * 128, __uint_as_float(v1[q]));
        tmem_ld_32x32b_x32(tmem + lane_base + kColDQ + 64, v0);
        tmem_ld_32x32b_x32(tmem + lane_base + kColDQ + 96, v1);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->dq_empty);
        if (second) {
          dst = a.dq_acc + r1 * 128 + d;
#pragma unroll
          for (int q = 0; q < 32; ++q) bwd::red_add_f32(dst + q * 128, __uint_as_float(v0[q]));
#pragma unroll
          for (int q = 0; q < 32; ++q)
            bwd::red_add_f32(dst + (32 + q) * 128, __uint_as_float(v1[q]));
        }
      }
    }
  }

  // ------------------------------------------------------------------ dK, dV epilogue
  // (dK takes the factor scale that dS left out)
  const bool any = g > 0;
  if (warp == kMmaWarp) {
    // every MMA issued has completed before TMEM can be released
    warp_mma_commit(&ctl->drain);
    wait(&ctl->drain, 0, ctl, a, 0x70, true);
    __syncwarp();
  } else if (warp == kListWarp) {
    if (any && ok) warp_mma_commit(&ctl->acc_full);
    warp_mma_commit(&ctl->drain2);
    wait(&ctl->drain2, 0, ctl, a, 0x71, true);
    __syncwarp();
  } else if (warp == kTmaWarp) {
    if (lane == 0) {  // every copy issued has landed before the CTA exits
      if (kv_issued) wait(&ctl->kv_full, 0, ctl, a, 0x72, true);
      if (fills0) wait(&ctl->ld_full[0], (fills0 - 1) & 1, ctl, a, 0x73, true);
      if (fills1) wait(&ctl->ld_full[1], (fills1 - 1) & 1, ctl, a, 0x73, true);
    }
    __syncwarp();
  } else if (warp < 8) {
    // thread = d column (TMEM lane of dV^T / dK^T), 64 keys of the block
    const int d = (warp & 3) * 32 + (int)lane;
    const bool is_dk = warp >= 4;
    const float sc = is_dk ? a.scale : 1.0f;
    uint16_t* dst = (is_dk ? a.dk : a.dv) + ((long long)bkv * a.Sk + 64 * kb) * 128 + d;
    bool have = false;
    if (any && ok) {
      have = wait_warp(&ctl->acc_full, 0, ctl, a, 0x74);
      tc_fence_after();
    }
    if (have || !any) {
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t v[32];
        if (have) {
          tmem_ld_32x32b_x32(tmem + lane_base + (is_dk ? kColDK : kColDV) + 32 * c, v);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = 0u;  // no query row attends this key block
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const uint32_t h = pack_bf16x2(__uint_as_float(v[j]) * sc, 0.0f);
          dst[(32 * c + j) * 128] = (uint16_t)(h & 0xFFFFu);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace bwd64
}  // namespace vsa
