// vsa_fwd_kernel.cuh -- the block-sparse attention forward kernel for sm_103a.
//
// What it computes: for every query row, softmax attention restricted to the keys of
// the key blocks its query block selects, with each key block's tail keys (positions
// >= variable_block_sizes[kb]) masked; out in bf16 and the base-2 log-sum-exp in fp32;
// rows with no attended key get out = +0 and lse = -FLT_MAX.  ("FastVideo
// block_sparse_attn_sm100a.py", module and is_supported docstrings; "TheRock rocke
// sparse_attention.py", module docstring and the two build_* kernels.)
//
// How (one persistent CTA per SM, 10 warps, warp-specialised):
//   warp 8        producer: per work item, turns the LUT rows (or the Jenga bitmap
//                 rows) into an ascending list of selected key blocks in shared memory
//                 -- an SMEM bitmap scatter followed by a ballot/popc compaction, so a
//                 repeated or out-of-range LUT entry can never cause a duplicate or an
//                 out-of-bounds copy -- then issues TMA copies of Q and of ONLY the
//                 selected K/V blocks into a 4-stage ring (mbarrier full/empty pairs).
//   warp 9        MMA issuer: S = Q K^T (both operands from SMEM) into a
//                 double-buffered TMEM S tile, then O += P V with P read from TMEM
//                 (P overwrites S in place as bf16) and O in a double-buffered TMEM
//                 accumulator.
//   warps 0-3     softmax: one thread per query row; loads its S row from TMEM,
//                 applies the tail-key / row-half mask, keeps a running max in the
//                 log2 domain and only rescales O and l when the max grows by more
//                 than 2^8 (the reference value may lag the true max; out = O/l and
//                 lse = m + log2 l are exact for any common reference), writes bf16 P.
//   warps 4-7     epilogue: out = O / l (or +0 for empty rows) staged in SMEM and
//                 written by a TMA store; lse = m + log2 l or the sentinel.
//
// Work item = 128 query rows (the M of one tcgen05 MMA):
//   block 128: one query block; one key tile = one selected key block (N = 128).
//   block 64 : an adjacent PAIR of query blocks (the pairing "FastVideo
//              block_sparse_attn_sm100a.py" describes: a CTA owns an adjacent pair of
//              query blocks).  The pair walks the sorted UNION of its two selections;
//              each union entry carries a 2-bit row-half mask, and rows of the query
//              block that did not select it see -inf.  Two union blocks form one key
//              tile (N = 128; the last tile of an odd union has N = 64).
#pragma once

#include <cuda.h>
#include <cstdint>

#include "sm103_ptx.cuh"

namespace vsa {

constexpr int kThreads = 320;
constexpr int kStages = 4;
constexpr int kMaxNb = 2048;
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // one second per wait
constexpr float kRescaleThreshold = 8.0f;         // log2 units: stale max allowed to lag 2^8

// shared-memory map (bytes from a 1024-aligned base)
constexpr uint32_t kQBytes = 128 * 128 * 2;      // one Q (or out staging) tile
constexpr uint32_t kTileBytes = 128 * 128 * 2;   // one K or V tile of up to 128 keys
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffKV = kOffQ + 2 * kQBytes;
constexpr uint32_t kOffList = kOffKV + kStages * kTileBytes;
constexpr uint32_t kOffBm = kOffList + 2 * kMaxNb * 4;
constexpr uint32_t kOffStats = kOffBm + 2 * kMaxNb;
constexpr uint32_t kOffCtl = kOffStats + 2 * 2 * 128 * 4;
constexpr uint32_t kCtlBytes = 1024;
constexpr uint32_t kSmemBytes = kOffCtl + kCtlBytes + 1024;  // + alignment slack

// TMEM columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;    // two S/P buffers of 128 columns
constexpr uint32_t kColO = 256;  // two O buffers of 128 columns

// device status codes (the low byte names the wait that gave up)
constexpr unsigned kErrTimeout = 0x100u;

struct SmemCtl {
  uint64_t q_full[2], q_empty[2];
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t list_full[2], list_empty[2];
  uint64_t s_full[2], p_full[2];
  uint64_t pv_done;
  uint64_t o_full[2], o_empty[2];
  uint64_t stats_full[2];
  uint64_t epi_bar[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int hdr_item[2];
  int hdr_n[2];
};
static_assert(sizeof(SmemCtl) <= kCtlBytes, "control block too large");

struct FwdArgs {
  const int32_t* q2k_idx;  // VSA
  const int32_t* q2k_num;
  const int32_t* vbs;
  const int8_t* bitmap;    // Jenga
  float* lse;              // may be null
  unsigned int* sched;     // null = static schedule; else {next item, CTAs done}
  unsigned int* status;    // device status word
  int H, S, nb, max_kv, n_items;
  float scale_log2;
};

// Bounded wait on an mbarrier phase.  Gives up after kWaitLimitNs (recording `code` in
// the device status word and raising the CTA's abort flag), or as soon as another role
// has raised the abort flag (unless `drain`: waits for copies / MMAs in flight still run
// to their own time limit so nothing is in flight when the CTA exits).
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, SmemCtl* ctl,
                                         unsigned* status, unsigned code, bool drain = false) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (!drain && *reinterpret_cast<volatile int*>(&ctl->abort_flag)) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      *reinterpret_cast<volatile int*>(&ctl->abort_flag) = 1;
      atomicCAS(status, 0u, kErrTimeout | code);
      return false;
    }
  }
}

// list entry: bits 0-15 key block, bits 16-17 row-half mask, bits 20-27 valid keys
__device__ __forceinline__ uint32_t make_entry(int kb, uint32_t halves, int valid) {
  return (uint32_t)kb | (halves << 16) | ((uint32_t)valid << 20);
}

template <int BLOCK, bool JENGA>
struct Cfg {
  static constexpr int kSub = (BLOCK == 64) ? 2 : 1;     // key blocks per key tile
  static constexpr int kPairs = (BLOCK == 64) ? 2 : 1;   // query blocks per work item
};

// ------------------------------------------------------------------------------------
// producer warp: work items, block lists, TMA copies
// ------------------------------------------------------------------------------------
template <int BLOCK, bool JENGA>
__device__ void producer_role(uint8_t* smem, SmemCtl* ctl, const FwdArgs& a,
                              const CUtensorMap* tq, const CUtensorMap* tk,
                              const CUtensorMap* tv) {
  using C = Cfg<BLOCK, JENGA>;
  const uint32_t lane = lane_id();
  uint8_t* bm0 = smem + kOffBm;
  uint8_t* bm1 = bm0 + kMaxNb;
  const uint64_t pol_kv = policy_evict_last();
  const uint64_t pol_q = policy_evict_first();
  uint32_t L = 0;  // K/V tiles loaded so far (ring position)
  uint32_t fills[kStages] = {0, 0, 0, 0};
  uint32_t qfills[2] = {0, 0};
  const int nb = a.nb;
  for (uint32_t it = 0;; ++it) {
    const uint32_t buf = it & 1;
    // ---- next work item
    int item;
    if (a.sched == nullptr) {
      const long long s = (long long)blockIdx.x + (long long)it * gridDim.x;
      item = s < a.n_items ? (int)s : -1;
    } else {
      unsigned got = 0;
      if (lane == 0) got = atomicAdd(&a.sched[0], 1u);
      got = __shfl_sync(0xffffffffu, got, 0);
      item = got < (unsigned)a.n_items ? (int)got : -1;
    }
    if (it >= 2 && !wait_bar(&ctl->list_empty[buf], ((it >> 1) + 1) & 1, ctl, a.status, 1)) break;
    uint32_t* list = reinterpret_cast<uint32_t*>(smem + kOffList) + buf * kMaxNb;
    int count = 0;
    int bh = 0, qa = 0;
    if (item >= 0) {
      const int items_per_bh = nb / C::kPairs;
      bh = item / items_per_bh;
      qa = (item - bh * items_per_bh) * C::kPairs;
      if (!JENGA) {
        // scatter the LUT rows of the item's query blocks into per-half byte maps
#pragma unroll
        for (int hf = 0; hf < C::kPairs; ++hf) {
          const long long row = (long long)bh * nb + qa + hf;
          int n = a.q2k_num[row];
          n = n < 0 ? 0 : (n > a.max_kv ? a.max_kv : n);
          const int32_t* lut = a.q2k_idx + row * a.max_kv;
          uint8_t* bm = hf ? bm1 : bm0;
          for (int s = lane; s < n; s += 32) {
            const int kb = lut[s];
            if (kb >= 0 && kb < nb) bm[kb] = 1;
          }
        }
        __syncwarp();
      }
      // ascending compaction of the selected blocks
      for (int base = 0; base < nb; base += 32) {
        const int kb = base + (int)lane;
        uint32_t h0 = 0, h1 = 0;
        if (kb < nb) {
          if (JENGA) {
            h0 = a.bitmap[(long long)qa * nb + kb] != 0;
            if (C::kPairs == 2) h1 = a.bitmap[(long long)(qa + 1) * nb + kb] != 0;
          } else {
            h0 = bm0[kb];
            if (C::kPairs == 2) h1 = bm1[kb];
          }
        }
        const uint32_t sel = h0 | h1;
        const uint32_t ballot = __ballot_sync(0xffffffffu, sel != 0);
        if (sel) {
          const int pos = count + __popc(ballot & ((1u << lane) - 1u));
          int valid = BLOCK;
          if (!JENGA) {
            valid = a.vbs[kb];
            valid = valid < 0 ? 0 : (valid > BLOCK ? BLOCK : valid);
          }
          const uint32_t halves = (C::kPairs == 2) ? (h0 | (h1 << 1)) : 3u;
          list[pos] = make_entry(kb, halves, valid);
          if (!JENGA) {
            bm0[kb] = 0;
            if (C::kPairs == 2) bm1[kb] = 0;
          }
        }
        count += __popc(ballot);
      }
      __syncwarp();
    }
    if (lane == 0) {
      ctl->hdr_item[buf] = item;
      ctl->hdr_n[buf] = count;
      mbar_arrive(&ctl->list_full[buf]);
    }
    __syncwarp();
    if (item < 0) break;

    // ---- Q tile (128 rows) of the item
    const int row0 = bh * a.S + qa * BLOCK;
    if (it >= 2 && !wait_bar(&ctl->q_empty[buf], ((it >> 1) + 1) & 1, ctl, a.status, 2)) break;
    uint8_t* qs = smem + kOffQ + buf * kQBytes;
    if (lane == 0) {
      mbar_arrive_expect_tx(&ctl->q_full[buf], kQBytes);
      tma_load_2d_hint(qs, tq, &ctl->q_full[buf], 0, row0, pol_q);
      tma_load_2d_hint(qs + kQBytes / 2, tq, &ctl->q_full[buf], 64, row0, pol_q);
    }
    qfills[buf]++;

    // ---- K/V tiles in the order the MMA warp consumes them: K0, K1, V0, K2, V1, ...
    const int n_tiles = (count + C::kSub - 1) / C::kSub;
    bool ok = true;
    for (int t = 0; t <= n_tiles && ok; ++t) {
#pragma unroll
      for (int which = 0; which < 2; ++which) {  // 0: K of tile t, 1: V of tile t-1
        const int tt = which == 0 ? t : t - 1;
        if (tt < 0 || tt >= n_tiles) continue;
        const uint32_t stage = L % kStages;
        if (L >= kStages &&
            !wait_bar(&ctl->kv_empty[stage], ((L / kStages) + 1) & 1, ctl, a.status, 3)) {
          ok = false;
          break;
        }
        const CUtensorMap* map = which == 0 ? tk : tv;
        uint8_t* dst = smem + kOffKV + stage * kTileBytes;
        const int e0 = tt * C::kSub;
        const int ne = (count - e0) < C::kSub ? (count - e0) : C::kSub;
        if (lane == 0) {
          mbar_arrive_expect_tx(&ctl->kv_full[stage], (uint32_t)ne * BLOCK * 128 * 2);
          for (int e = 0; e < ne; ++e) {
            const int kb = (int)(list[e0 + e] & 0xFFFFu);
            const int krow = bh * a.S + kb * BLOCK;
            // d-halves are separate [128 rows][64] sub-tiles; block e fills rows e*BLOCK..
            tma_load_2d_hint(dst + e * BLOCK * 128, map, &ctl->kv_full[stage], 0, krow, pol_kv);
            tma_load_2d_hint(dst + kTileBytes / 2 + e * BLOCK * 128, map, &ctl->kv_full[stage],
                             64, krow, pol_kv);
          }
        }
        fills[stage]++;
        ++L;
      }
    }
    if (!ok) break;
  }
  // drain: every copy this warp issued has landed before the CTA can exit
  for (int s = 0; s < kStages; ++s)
    if (fills[s]) wait_bar(&ctl->kv_full[s], (fills[s] - 1) & 1, ctl, a.status, 4, true);
  for (int b = 0; b < 2; ++b)
    if (qfills[b]) wait_bar(&ctl->q_full[b], (qfills[b] - 1) & 1, ctl, a.status, 5, true);
}

// ------------------------------------------------------------------------------------
// MMA warp (one thread issues)
// ------------------------------------------------------------------------------------
template <int BLOCK, bool JENGA>
__device__ void mma_role(uint8_t* smem, SmemCtl* ctl, const FwdArgs& a, uint32_t tmem) {
  using C = Cfg<BLOCK, JENGA>;
  constexpr uint32_t kIdescS128 = idesc_bf16_f32(128, 128, false, false);
  constexpr uint32_t kIdescS64 = idesc_bf16_f32(128, 64, false, false);
  constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 128, false, true);
  uint32_t L = 0, g = 0;
  for (uint32_t it = 0;; ++it) {
    const uint32_t buf = it & 1;
    if (!wait_bar(&ctl->list_full[buf], (it >> 1) & 1, ctl, a.status, 10)) break;
    const int item = ctl->hdr_item[buf];
    const int count = ctl->hdr_n[buf];
    mbar_arrive(&ctl->list_empty[buf]);
    if (item < 0) break;
    if (it >= 2 && !wait_bar(&ctl->o_empty[buf], ((it >> 1) + 1) & 1, ctl, a.status, 11)) break;
    if (!wait_bar(&ctl->q_full[buf], (it >> 1) & 1, ctl, a.status, 12)) break;
    tc_fence_after();
    const uint32_t qaddr = smem_addr(smem + kOffQ + buf * kQBytes);
    const uint32_t tO = tmem + kColO + buf * 128;
    const int n_tiles = (count + C::kSub - 1) / C::kSub;
    bool ok = true;
    for (int t = 0; t <= n_tiles && ok; ++t) {
      if (t < n_tiles) {  // S_t = Q K_t^T
        const uint32_t gg = g + t;
        const uint32_t stage = L % kStages;
        if (!wait_bar(&ctl->kv_full[stage], (L / kStages) & 1, ctl, a.status, 13)) { ok = false; break; }
        tc_fence_after();
        const int ne = (count - t * C::kSub) < C::kSub ? (count - t * C::kSub) : C::kSub;
        const uint32_t idesc = (ne * BLOCK == 128) ? kIdescS128 : kIdescS64;
        const uint32_t kaddr = smem_addr(smem + kOffKV + stage * kTileBytes);
        const uint32_t tS = tmem + kColS + (gg & 1) * 128;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t off = (k >> 2) * (kTileBytes / 2) + (k & 3) * 32;
          mma_ss(tS, smem_desc_sw128(qaddr + off, 16, 1024), smem_desc_sw128(kaddr + off, 16, 1024),
                 idesc, k > 0);
        }
        mma_commit(&ctl->kv_empty[stage]);
        mma_commit(&ctl->s_full[gg & 1]);
        ++L;
      }
      if (t >= 1) {  // O += P_{t-1} V_{t-1}
        const int tp = t - 1;
        const uint32_t gg = g + tp;
        if (!wait_bar(&ctl->p_full[gg & 1], (gg >> 1) & 1, ctl, a.status, 14)) { ok = false; break; }
        const uint32_t stage = L % kStages;
        if (!wait_bar(&ctl->kv_full[stage], (L / kStages) & 1, ctl, a.status, 15)) { ok = false; break; }
        tc_fence_after();
        const int ne = (count - tp * C::kSub) < C::kSub ? (count - tp * C::kSub) : C::kSub;
        const int ksteps = ne * BLOCK / 16;
        const uint32_t vaddr = smem_addr(smem + kOffKV + stage * kTileBytes);
        const uint32_t tP = tmem + kColS + (gg & 1) * 128;
        for (int k = 0; k < ksteps; ++k) {
          mma_ts(tO, tP + k * 8, smem_desc_sw128(vaddr + k * 2048, kTileBytes / 2, 1024), kIdescPV,
                 (tp > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(&ctl->kv_empty[stage]);
        mma_commit(&ctl->pv_done);
        ++L;
      }
    }
    if (!ok) break;
    mma_commit(&ctl->o_full[buf]);
    g += n_tiles;
  }
  // every MMA issued has completed before TMEM can be released
  mma_commit(&ctl->drain);
  wait_bar(&ctl->drain, 0, ctl, a.status, 16, true);
}

// ------------------------------------------------------------------------------------
// softmax warpgroup (warps 0-3): thread = query row of the 128-row tile
// ------------------------------------------------------------------------------------
template <int NK>
__device__ __forceinline__ void softmax_tile(uint32_t tS, int lim0, int lim1, int kps, float sl2,
                                             float& m_run, float& l_run, float& alpha) {
  uint32_t r[NK];
#pragma unroll
  for (int c = 0; c < NK / 32; ++c)
    tmem_ld_32x32b_x32(tS + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&r[c * 32]));
  tmem_wait_ld();
  float s[NK];
#pragma unroll
  for (int j = 0; j < NK; ++j) s[j] = __uint_as_float(r[j]);
  if (lim0 < kps || (NK > kps && lim1 < kps)) {
#pragma unroll
    for (int j = 0; j < NK; ++j) {
      const int lim = (j < kps) ? lim0 : lim1;
      const int jj = (j < kps) ? j : j - kps;
      if (jj >= lim) s[j] = -INFINITY;
    }
  }
  // row max (pairwise tree for ILP)
  float mx[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) mx[i] = s[i];
#pragma unroll
  for (int j = 8; j < NK; ++j) mx[j & 7] = fmaxf(mx[j & 7], s[j]);
  const float mraw = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                           fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
  const float m_tile = mraw * sl2;
  alpha = 1.0f;
  if (m_tile > m_run + kRescaleThreshold) {
    if (m_run != -INFINITY) alpha = fast_exp2(m_run - m_tile);
    m_run = m_tile;
  }
  const float neg = (m_run == -INFINITY) ? 0.0f : -m_run;
#pragma unroll
  for (int j = 0; j < NK; ++j) s[j] = fast_exp2(fmaf(s[j], sl2, neg));
  // P is rounded to bf16 for the PV MMA; l sums exactly those rounded weights, so the
  // weights applied to V are normalised consistently (with a lagging reference max the
  // unrounded sum would leave up to ~2^-8 relative mismatch on dominant keys).
  uint32_t pk[NK / 2];
  float sum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < NK / 2; ++i) {
    pk[i] = pack_bf16x2(s[2 * i], s[2 * i + 1]);
    sum[i & 3] += __uint_as_float(pk[i] << 16) + __uint_as_float(pk[i] & 0xFFFF0000u);
  }
  l_run = l_run * alpha + ((sum[0] + sum[1]) + (sum[2] + sum[3]));
#pragma unroll
  for (int c = 0; c < NK / 64; ++c)
    tmem_st_32x32b_x32(tS + c * 32, *reinterpret_cast<const uint32_t(*)[32]>(&pk[c * 32]));
}

template <int BLOCK, bool JENGA>
__device__ void softmax_role(uint8_t* smem, SmemCtl* ctl, const FwdArgs& a, uint32_t tmem) {
  using C = Cfg<BLOCK, JENGA>;
  constexpr int kps = BLOCK;  // keys per key block
  const int row = threadIdx.x;             // 0..127
  const uint32_t warp = threadIdx.x >> 5;  // 0..3
  const uint32_t lane_base = (warp * 32) << 16;
  const uint32_t half = (BLOCK == 64) ? (uint32_t)(row >> 6) : 0u;
  float* stat_m = reinterpret_cast<float*>(smem + kOffStats);
  float* stat_l = stat_m + 2 * 128;
  uint32_t g = 0;
  for (uint32_t it = 0;; ++it) {
    const uint32_t buf = it & 1;
    if (!wait_bar(&ctl->list_full[buf], (it >> 1) & 1, ctl, a.status, 20)) break;
    const int item = ctl->hdr_item[buf];
    const int count = ctl->hdr_n[buf];
    if (item < 0) break;
    const uint32_t* list = reinterpret_cast<const uint32_t*>(smem + kOffList) + buf * kMaxNb;
    const uint32_t tO = tmem + kColO + buf * 128 + lane_base;
    const int n_tiles = (count + C::kSub - 1) / C::kSub;
    float m_run = -INFINITY, l_run = 0.0f;
    bool ok = true;
    for (int t = 0; t < n_tiles; ++t) {
      const uint32_t gg = g + t;
      const int e0 = t * C::kSub;
      const int ne = (count - e0) < C::kSub ? (count - e0) : C::kSub;
      const uint32_t en0 = list[e0];
      const int lim0 = ((en0 >> (16 + half)) & 1u) ? (int)((en0 >> 20) & 0xFFu) : 0;
      int lim1 = kps;
      if (ne > 1) {
        const uint32_t en1 = list[e0 + 1];
        lim1 = ((en1 >> (16 + half)) & 1u) ? (int)((en1 >> 20) & 0xFFu) : 0;
      }
      if (!wait_bar(&ctl->s_full[gg & 1], (gg >> 1) & 1, ctl, a.status, 21)) { ok = false; break; }
      tc_fence_after();
      const uint32_t tS = tmem + kColS + (gg & 1) * 128 + lane_base;
      float alpha;
      if (ne * BLOCK == 128)
        softmax_tile<128>(tS, lim0, lim1, kps, a.scale_log2, m_run, l_run, alpha);
      else
        softmax_tile<64>(tS, lim0, lim1, kps, a.scale_log2, m_run, l_run, alpha);
      // O rescale when this row's reference max moved (warp-uniform TMEM access)
      if (__any_sync(0xffffffffu, alpha != 1.0f)) {
        if (!wait_bar(&ctl->pv_done, (gg - 1) & 1, ctl, a.status, 22)) { ok = false; break; }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(tO + c * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
          tmem_st_32x32b_x32(tO + c * 32, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if ((threadIdx.x & 31) == 0) mbar_arrive(&ctl->p_full[gg & 1]);
    }
    if (!ok) break;
    g += n_tiles;
    stat_m[buf * 128 + row] = m_run;
    stat_l[buf * 128 + row] = l_run;
    __syncwarp();
    if ((threadIdx.x & 31) == 0) {
      mbar_arrive(&ctl->stats_full[buf]);
      mbar_arrive(&ctl->list_empty[buf]);
    }
  }
}

// ------------------------------------------------------------------------------------
// epilogue warpgroup (warps 4-7)
// ------------------------------------------------------------------------------------
template <int BLOCK, bool JENGA>
__device__ void epilogue_role(uint8_t* smem, SmemCtl* ctl, const FwdArgs& a, uint32_t tmem,
                              const CUtensorMap* to) {
  using C = Cfg<BLOCK, JENGA>;
  const int row = threadIdx.x - 128;       // 0..127
  const uint32_t warp = threadIdx.x >> 5;  // 4..7
  const uint32_t lane_base = ((warp & 3) * 32) << 16;
  const float* stat_m = reinterpret_cast<const float*>(smem + kOffStats);
  const float* stat_l = stat_m + 2 * 128;
  const bool leader = threadIdx.x == 128;
  for (uint32_t it = 0;; ++it) {
    const uint32_t buf = it & 1;
    if (!wait_bar(&ctl->list_full[buf], (it >> 1) & 1, ctl, a.status, 30)) break;
    const int item = ctl->hdr_item[buf];
    const int count = ctl->hdr_n[buf];
    if (item < 0) break;
    const int items_per_bh = a.nb / C::kPairs;
    const int bh = item / items_per_bh;
    const int qa = (item - bh * items_per_bh) * C::kPairs;
    const int row0 = bh * a.S + qa * BLOCK;
    if (!wait_bar(&ctl->stats_full[buf], (it >> 1) & 1, ctl, a.status, 31)) break;
    if (!wait_bar(&ctl->o_full[buf], (it >> 1) & 1, ctl, a.status, 32)) break;
    tc_fence_after();
    const float m = stat_m[buf * 128 + row];
    const float l = stat_l[buf * 128 + row];
    const bool has = l > 0.0f;
    const float inv = has ? 1.0f / l : 0.0f;
    uint8_t* qs = smem + kOffQ + buf * kQBytes;
    const uint32_t tO = tmem + kColO + buf * 128 + lane_base;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      uint32_t o[32];
      if (count > 0) {
        tmem_ld_32x32b_x32(tO + c * 32, o);
        tmem_wait_ld();
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float x0 = 0.0f, x1 = 0.0f;
          if (has) {
            x0 = __uint_as_float(o[8 * i + 2 * j]) * inv;
            x1 = __uint_as_float(o[8 * i + 2 * j + 1]) * inv;
          }
          w[j] = pack_bf16x2(x0, x1);
        }
        const uint32_t chunk = (uint32_t)((c & 1) * 4 + i);     // 16-byte chunk in the 128B row
        const uint32_t phys = chunk ^ (uint32_t)(row & 7);      // 128-byte swizzle
        uint8_t* dst = qs + (c >> 1) * (kQBytes / 2) + row * 128 + phys * 16;
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(smem_addr(dst)), "r"(w[0]),
                     "r"(w[1]), "r"(w[2]), "r"(w[3])
                     : "memory");
      }
    }
    if (a.lse != nullptr) a.lse[(long long)row0 + row] = has ? m + log2f(l) : -3.402823466e+38f;
    tc_fence_before();
    fence_proxy_async_smem();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) {
      // O, the row statistics and the list header of this buffer are no longer needed
      mbar_arrive(&ctl->o_empty[buf]);
      mbar_arrive(&ctl->list_empty[buf]);
      mbar_arrive(&ctl->epi_bar[buf]);
    }
    if (leader) {
      if (!wait_bar(&ctl->epi_bar[buf], (it >> 1) & 1, ctl, a.status, 33)) break;
      tma_store_2d(to, qs, 0, row0);
      tma_store_2d(to, qs + kQBytes / 2, 64, row0);
      bulk_commit_group();
      bulk_wait_group_read0();
      mbar_arrive(&ctl->q_empty[buf]);
    }
  }
  if (leader) bulk_wait_group0();
}

// ------------------------------------------------------------------------------------
template <int BLOCK, bool JENGA>
__global__ void __launch_bounds__(kThreads, 1)
    bsa_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
                   const FwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  SmemCtl* ctl = reinterpret_cast<SmemCtl*>(smem + kOffCtl);
  const uint32_t warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctl->q_full[i], 1);
      mbar_init(&ctl->q_empty[i], 1);
      mbar_init(&ctl->list_full[i], 1);
      mbar_init(&ctl->list_empty[i], 9);
      mbar_init(&ctl->s_full[i], 1);
      mbar_init(&ctl->p_full[i], 4);
      mbar_init(&ctl->o_full[i], 1);
      mbar_init(&ctl->o_empty[i], 4);
      mbar_init(&ctl->stats_full[i], 4);
      mbar_init(&ctl->epi_bar[i], 4);
    }
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&ctl->kv_full[i], 1);
      mbar_init(&ctl->kv_empty[i], 1);
    }
    mbar_init(&ctl->pv_done, 1);
    mbar_init(&ctl->drain, 1);
    ctl->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 8) {
    // the per-half byte maps start (and are always left) all zero
    uint32_t* bm = reinterpret_cast<uint32_t*>(smem + kOffBm);
    for (int i = lane_id(); i < 2 * kMaxNb / 4; i += 32) bm[i] = 0;
    if (lane_id() == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      tma_prefetch_desc(&to);
    }
  }
  if (warp == 9) {
    tmem_alloc(&ctl->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  if (warp < 4) {
    softmax_role<BLOCK, JENGA>(smem, ctl, a, tmem);
  } else if (warp < 8) {
    epilogue_role<BLOCK, JENGA>(smem, ctl, a, tmem, &to);
  } else if (warp == 8) {
    producer_role<BLOCK, JENGA>(smem, ctl, a, &tq, &tk, &tv);
  } else {
    if (lane_id() == 0) mma_role<BLOCK, JENGA>(smem, ctl, a, tmem);
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) tmem_dealloc(tmem, kTmemCols);
  // dynamic schedule: the last CTA to finish returns the counters to zero
  if (a.sched != nullptr && threadIdx.x == 0) {
    __threadfence();
    const unsigned done = atomicAdd(&a.sched[1], 1u);
    if (done == gridDim.x - 1) {
      atomicExch(&a.sched[0], 0u);
      atomicExch(&a.sched[1], 0u);
    }
  }
}

}  // namespace vsa
