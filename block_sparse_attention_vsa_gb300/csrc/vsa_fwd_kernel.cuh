// vsa_fwd_kernel.cuh -- the block-sparse attention forward kernel for sm_103a.
//
// What it computes: for every query row, softmax attention restricted to the keys of
// the key blocks its query block selects, with each key block's tail keys (positions
// >= variable_block_sizes[kb]) masked; out in bf16 and the base-2 log-sum-exp in fp32;
// rows with no attended key get out = +0 and lse = -FLT_MAX.  ("FastVideo
// block_sparse_attn_sm100a.py", module and is_supported docstrings; "TheRock rocke
// sparse_attention.py", module docstring and the two build_* kernels.)
//
// Work item = 128 query rows (the M of one tcgen05 MMA):
//   block 128: one query block; one key tile = one selected key block (N = 128).
//   block 64 : an adjacent PAIR of query blocks (the pairing "FastVideo
//              block_sparse_attn_sm100a.py" describes: a CTA owns an adjacent pair of
//              query blocks).  The pair walks the sorted UNION of its two selections;
//              each union entry carries a 2-bit row-half mask, and rows of the query
//              block that did not select it see -inf.  Two union blocks form one key
//              tile (N = 128; the last tile of an odd union has N = 64).
//
// Structure: one persistent CTA per SM, 12 warps.
//   warp 10     lists: per work item, one item ahead of its use, turns the LUT rows (or
//               block-map rows) into the list of selected key blocks -- an SMEM byte-map
//               scatter then a ballot/popc compaction, so repeated or out-of-range LUT
//               entries can never cause a duplicate or an out-of-bounds copy.  Block-64
//               lists put blocks only one query block selects in alternating pairs first
//               (see build_list).  Lists are double-buffered.
//   warp 8      TMA (one thread): Q (double-buffered across items) and ONLY the
//               selected K/V blocks into a 4-stage ring, in the order the MMA warp
//               consumes them.
//   warp 9      MMA issuer (one thread): S_g = Q K_g^T into TMEM S buffer g%2 (g counts
//               key tiles across items), then, per key half w, O_w += P_g[:, 64w:64w+64]
//               V_g[64w:64w+64, :] with P read from TMEM.  Issue order QK0, QK1, PV0,
//               QK2, PV1, ..., so QK_{t+1} runs while P_t is computed.  Two commits per
//               tile release the K and the V ring stage (see SmemCtl).
//   warps 0-3   softmax warpgroup 0: keys 0-63 of every key tile;
//   warps 4-7   softmax warpgroup 1: keys 64-127 of every key tile.  One thread per
//               query row; each warpgroup keeps its own running max m (log2 domain,
//               allowed to lag the true max by up to 2^32 before O and l are rescaled),
//               row sums and O accumulator, so the two never synchronise inside the key
//               loop.  After the item they merge (m, l, O) of both halves and each
//               warpgroup normalises, stages (in the item's Q buffer) and TMA-stores
//               one 64-column half of the output; warpgroup 0 writes lse.  The store
//               leader releases that Q buffer only after the next item's first tile,
//               so the store's read of SMEM never holds up an item boundary.
//   warp 11     at the start, copies variable_block_sizes (clamped) into SMEM for the list
//               warp's compaction; then idle.
// TMEM (512 columns): S0, S1 at columns 0, 128 (warpgroup w reads S columns 64w..64w+63
// and writes its bf16 P over the first 32 of them); O0, O1 at 256, 384.
// Every mbarrier wait is bounded; a wait that runs out records a code in the device
// status word, raises the CTA's abort flag and every role returns.  Waits that a whole
// warp goes on from into warp-collective instructions (the list and softmax warps) are
// warp votes, so a warp never splits; the TMA and MMA roles run on one thread each.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "sm103_ptx.cuh"

namespace vsa {

constexpr int kThreads = 384;
constexpr int kStages = 4;
constexpr int kMaxNb = 2048;
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // one second per wait
// log2 units: the running max may lag the true one by up to 2^32 before O and l are
// rescaled (each rescale waits for the previous PV).  P <= 2^32 is in range for bf16;
// with at most 2048 * 128 keys per row (2048 blocks of 128), l <= 2^50 and
// |O| <= 2^50 max|v| stay finite in fp32 for |v| < 3e23.
constexpr float kRescaleThreshold = 32.0f;
constexpr uint32_t kSoftmaxRegs = 216;            // per thread, softmax warpgroups
constexpr uint32_t kOtherRegs = 56;               // per thread, TMA / MMA / list warps
// registers the launch must provide for the re-balancing above (checked on the host)
constexpr uint32_t kRegPoolNeeded = 256 * kSoftmaxRegs + 128 * kOtherRegs;

// shared-memory map (bytes from a 1024-aligned base)
constexpr uint32_t kTileBytes = 128 * 128 * 2;  // a Q / out-staging / K / V tile
constexpr uint32_t kOffQ = 0;                   // Q[2] (double-buffered across items)
constexpr uint32_t kOffKV = 2 * kTileBytes;     // K/V ring [kStages]
constexpr uint32_t kOffList = kOffKV + kStages * kTileBytes;  // list[2][kMaxNb] u32
constexpr uint32_t kOffBm = kOffList + 2 * kMaxNb * 4;       // byte maps [2][kMaxNb]
constexpr uint32_t kOffStats = kOffBm + 2 * kMaxNb;          // [item parity][wg][3][128] f32
constexpr uint32_t kStatsBytes = 2 * 2 * 3 * 128 * 4;
constexpr uint32_t kOffVbs = kOffStats + kStatsBytes;  // valid keys per key block [kMaxNb] u8
constexpr uint32_t kOffCtl = kOffVbs + kMaxNb;
constexpr uint32_t kCtlBytes = 1024;
constexpr uint32_t kSmemBytes = kOffCtl + kCtlBytes + 1024;  // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "forward SMEM");
static_assert(kOffCtl % 8 == 0, "control block alignment");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;    // S0, S1
constexpr uint32_t kColO = 256;  // O0, O1

constexpr unsigned kErrTimeout = 0x100u;  // | code of the wait that gave up

struct SmemCtl {
  uint64_t list_full[2], list_empty[2];
  // q_full[b]: Q of an item landed in buffer b.  q_empty[b]: both store leaders' output
  // stores have read buffer b (the output is staged in the item's Q buffer), arrived one
  // tile into the next item, so the TMA warp can load the item after next.
  uint64_t q_full[2], q_empty[2];
  // kv_full[s]: ring stage s holds its tile.  kv_empty[s]: the MMAs that read the
  // stage's tile have completed.  The MMA warp commits kv_empty right after a tile's QK
  // (K stage) and after its PV (V stage), so the same phases also tell the softmax warps
  // that S is ready (K stage) and that O is up to date (V stage).  A stage is reused
  // every kStages ring positions, and the tile loaded there next cannot be consumed
  // before every waiter has moved on, so no waiter is ever two phases behind.
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t p_full[4];   // [2 b + w]: the 4 warps of softmax warpgroup w have written their
                        // P into S buffer b (per buffer, so a warp running a tile ahead can
                        // never complete the previous tile's phase; per warpgroup, so each
                        // key half's PV starts as soon as its own P is there)
  uint64_t o_full, o_empty;
  uint64_t stats_bar[2];
  uint64_t epi_bar[2];
  uint64_t drain;
  uint64_t vbs_ready;  // warp 11 has copied variable_block_sizes into SMEM
  uint64_t never;   // completed by nobody (the timeout test hook waits on it)
  int hdr_item[2];  // work unit (item * n_splits + split), -1 = no more work
  int hdr_n[2];     // list entries of the unit
  int hdr_off[2];   // index of the unit's first entry in the item's list
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(SmemCtl) <= kCtlBytes, "control block too large");

// Shapes: q / out [B, Hq, Sq, 128], k / v [B, Hkv, Sk, 128]; query head hq of batch b
// reads key/value head b*Hkv + hq / group.  nbq = Sq / BLOCK query blocks, nbk = Sk / BLOCK
// key blocks; a work item is one query block (BLOCK 128) or an adjacent pair (BLOCK 64,
// the last item of a head holding a single block when nbq is odd).
struct FwdArgs {
  const int32_t* q2k_idx;  // LUT mode: [B*Hq*nbq, max_kv]
  const int32_t* q2k_num;  //           [B*Hq*nbq]
  const int32_t* vbs;      // [nbk] valid keys per key block, or null = every block full
  const int8_t* bitmap;    // bitmap mode: [nbq, nbk] rows, (b*Hq + hq) * bitmap_bh_stride apart
  long long bitmap_bh_stride;  // 0 = one map shared by every (b, hq)
  float* lse;              // [B*Hq*Sq] or null
  unsigned int* sched;     // null = static schedule; else {next item, CTAs done}
  unsigned int* status;    // device status word
  float* part;             // split-KV partials [n_items][kPartFloats], or null
  int Hq, Hkv, group, Sq, Sk, nbq, nbk, max_kv, n_items, items_per_bh;
  int n_splits;            // key-tile ranges per item; n_items counts units (item, range)
  float scale_log2;
  unsigned long long wait_ns;  // limit of the waits that are not drains (kWaitLimitNs)
  int stall;               // test hook: the MMA warp first waits on a barrier nobody completes
};

// Split-KV partial of one unit: O [128 rows][128] fp32, unnormalised relative to the
// row's m, then m, l_round, l_exact per row (m = -inf and l = 0 for a row that attended
// nothing in the unit's range).
constexpr int kPartFloats = 128 * 128 + 3 * 128;

// Bounded wait on an mbarrier phase.  Gives up after the launch's limit a.wait_ns
// (recording `code` in the device status word and raising the CTA's abort flag), or as
// soon as another role has raised the abort flag -- unless `drain`: a wait for copies /
// MMAs still in flight always runs to the full kWaitLimitNs, so nothing is in flight
// when the CTA exits.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, SmemCtl* ctl,
                                         const FwdArgs& a, unsigned code, bool drain = false) {
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

// The same wait by every lane of a warp that goes on to warp-collective instructions
// (tcgen05.ld/st .sync.aligned, shuffles, votes): the warp proceeds only if every lane saw
// the phase complete, so giving up can never leave part of a warp behind.
__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity, SmemCtl* ctl,
                                          const FwdArgs& a, unsigned code) {
  const bool w = wait_bar(bar, parity, ctl, a, code);
  return __all_sync(0xffffffffu, w);
}

// list entry: bits 0-15 key block, bits 16-17 row-half mask, bits 20-27 valid keys
__device__ __forceinline__ uint32_t make_entry(int kb, uint32_t halves, int valid) {
  return (uint32_t)kb | (halves << 16) | ((uint32_t)valid << 20);
}
// valid keys of an entry for a row in query half `half` (0 if that half did not select it)
__device__ __forceinline__ int entry_limit(uint32_t e, uint32_t half) {
  return ((e >> (16 + half)) & 1u) ? (int)((e >> 20) & 0xFFu) : 0;
}

template <int BLOCK>
struct Cfg {
  static constexpr int kSub = (BLOCK == 64) ? 2 : 1;    // key blocks per key tile
  static constexpr int kPairs = (BLOCK == 64) ? 2 : 1;  // query blocks per work item
};

// ------------------------------------------------------------------------------------
// list warp (work items, block lists) and TMA warp (copies)
// ------------------------------------------------------------------------------------
struct ItemHead {
  int item, count, bh, qa;
};

// Pick the CTA's it-th work item, build its key-block list into list buffer it & 1 and
// publish the header (item -1 = no more work).  `ok` turns false if a wait gave up.
template <int BLOCK, bool JENGA>
__device__ ItemHead build_list(uint8_t* smem, SmemCtl* ctl, const FwdArgs& a, uint32_t it,
                               bool& ok) {
  using C = Cfg<BLOCK>;
  const uint32_t lane = lane_id();
  uint8_t* bm0 = smem + kOffBm;
  uint8_t* bm1 = bm0 + kMaxNb;
  const int nb = a.nbk;
  const uint32_t buf = it & 1;
  ItemHead h{-1, 0, 0, 0};
  if (a.sched == nullptr) {
    const long long s = (long long)blockIdx.x + (long long)it * gridDim.x;
    h.item = s < a.n_items ? (int)s : -1;
  } else {
    unsigned got = 0;
    if (lane == 0) got = atomicAdd(&a.sched[0], 1u);
    got = __shfl_sync(0xffffffffu, got, 0);
    h.item = got < (unsigned)a.n_items ? (int)got : -1;
  }
  if (it >= 2 && !wait_warp(&ctl->list_empty[buf], ((it >> 1) + 1) & 1, ctl, a, 1)) {
    ok = false;
    return h;
  }
  uint32_t* list = reinterpret_cast<uint32_t*>(smem + kOffList) + buf * kMaxNb;
  int count = 0, off = 0;
  if (h.item >= 0) {
    const int item = h.item / a.n_splits;
    h.bh = item / a.items_per_bh;
    h.qa = (item - h.bh * a.items_per_bh) * C::kPairs;
    const bool pair = C::kPairs == 2 && h.qa + 1 < a.nbq;  // the second query block exists
    // the item's selection as byte maps (which start, and are always left, all zero)
    if (!JENGA) {
      // The rows' counts and their first 128 slots are loaded together, before any store
      // to the byte maps (a store there may not be moved above a later load, so loads
      // interleaved with stores would each wait a round trip).  Slots past a row's count
      // lie inside the caller's LUT row and are read but never used.
      const long long row0 = (long long)h.bh * a.nbq + h.qa;
      const int rows = (C::kPairs == 2 && pair) ? 2 : 1;
      const int32_t* lut0 = a.q2k_idx + row0 * a.max_kv;
      const int32_t* lut1 = lut0 + a.max_kv;
      const int cnt = (int)lane < rows ? __ldg(a.q2k_num + row0 + lane) : 0;
      int kb0[4], kb1[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int s = 32 * j + (int)lane;
        kb0[j] = s < a.max_kv ? __ldg(lut0 + s) : -1;
        kb1[j] = (rows == 2 && s < a.max_kv) ? __ldg(lut1 + s) : -1;
      }
      int n0 = __shfl_sync(0xffffffffu, cnt, 0);
      int n1 = __shfl_sync(0xffffffffu, cnt, 1);
      n0 = n0 < 0 ? 0 : (n0 > a.max_kv ? a.max_kv : n0);
      n1 = rows == 2 ? (n1 < 0 ? 0 : (n1 > a.max_kv ? a.max_kv : n1)) : 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int s = 32 * j + (int)lane;
        if (s < n0 && kb0[j] >= 0 && kb0[j] < nb) bm0[kb0[j]] = 1;
        if (s < n1 && kb1[j] >= 0 && kb1[j] < nb) bm1[kb1[j]] = 1;
      }
      // slots 128 and on (a LUT wider than 128), four loads per lane at a time
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int n = hf ? n1 : n0;
        const int32_t* lut = hf ? lut1 : lut0;
        uint8_t* bm = hf ? bm1 : bm0;
        for (int s0 = 128; s0 < n; s0 += 128) {
          int kbv[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int s = s0 + 32 * j + (int)lane;
            kbv[j] = s < n ? __ldg(lut + s) : -1;
          }
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (kbv[j] >= 0 && kbv[j] < nb) bm[kbv[j]] = 1;
        }
      }
    } else {
      const int8_t* mrow = a.bitmap + h.bh * a.bitmap_bh_stride + (long long)h.qa * nb;
      for (int base = 0; base < nb; base += 128) {
        int8_t v0[4], v1[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int kb = base + 32 * j + (int)lane;
          v0[j] = kb < nb ? mrow[kb] : 0;
          v1[j] = (pair && kb < nb) ? mrow[nb + kb] : 0;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int kb = base + 32 * j + (int)lane;
          if (kb < nb) {
            bm0[kb] = v0[j] != 0;
            if (C::kPairs == 2) bm1[kb] = v1[j] != 0;
          }
        }
      }
    }
    __syncwarp();
    // which query block(s) select key block kb (bit 0: the first, bit 1: the second)
    auto selected = [&](int kb) -> uint32_t {
      if (kb >= nb) return 0u;
      return (uint32_t)bm0[kb] | (C::kPairs == 2 ? (uint32_t)bm1[kb] << 1 : 0u);
    };
    // (the CTA's copy of variable_block_sizes, already clamped to [0, BLOCK])
    auto valid_keys = [&](int kb) -> int {
      return a.vbs != nullptr ? (int)smem[kOffVbs + kb] : BLOCK;
    };
    // the block sizes the compaction reads come from warp 11's copy (block-64 pairs wait
    // after their counting pass, which does not read them)
    auto sizes_ready = [&]() -> bool {
      return it != 0 || a.vbs == nullptr || wait_warp(&ctl->vbs_ready, 0, ctl, a, 9);
    };
    const uint32_t below = (1u << lane) - 1u;
    if (C::kPairs == 1 && !sizes_ready()) {
      ok = false;
      return h;
    }
    if (C::kPairs == 1) {
      // ascending compaction
      for (int base = 0; base < nb; base += 32) {
        const int kb = base + (int)lane;
        const uint32_t sel = selected(kb);
        const int valid = kb < nb ? valid_keys(kb) : 0;
        const uint32_t ballot = __ballot_sync(0xffffffffu, sel != 0);
        if (sel) list[count + __popc(ballot & below)] = make_entry(kb, 3u, valid);
        count += __popc(ballot);
      }
    } else {
      // Block-64 pairs.  A key tile is two consecutive entries, one per softmax
      // warpgroup; the first query block's rows sit on two SM sub-partitions, the
      // second's on the other two.  A tile pairing a block only the first query block
      // selected (X) with one only the second selected (Y) gives every sub-partition one
      // busy softmax warp instead of two busy and two idle, so the list is laid out as
      // min(|X|, |Y|) XY tiles first, then the remaining X or Y, then the blocks both
      // select (each kind ascending).  The order changes only the summation order.
      int nx = 0, ny = 0;
      for (int base = 0; base < nb; base += 32) {
        const uint32_t sel = selected(base + (int)lane);
        nx += __popc(__ballot_sync(0xffffffffu, sel == 1u));
        ny += __popc(__ballot_sync(0xffffffffu, sel == 2u));
      }
      if (!sizes_ready()) {
        ok = false;
        return h;
      }
      const int xy = nx < ny ? nx : ny;
      const int rest = (nx - xy) + (ny - xy);
      int cx = 0, cy = 0, cb = 0;
      for (int base = 0; base < nb; base += 32) {
        const int kb = base + (int)lane;
        const uint32_t sel = selected(kb);
        const int valid = kb < nb ? valid_keys(kb) : 0;
        const uint32_t bx = __ballot_sync(0xffffffffu, sel == 1u);
        const uint32_t by = __ballot_sync(0xffffffffu, sel == 2u);
        const uint32_t bb = __ballot_sync(0xffffffffu, sel == 3u);
        // this block's rank among the blocks of its kind so far (selects, no branches)
        const uint32_t mine = sel == 1u ? bx : (sel == 2u ? by : bb);
        const int i = (sel == 1u ? cx : (sel == 2u ? cy : cb)) + __popc(mine & below);
        const int single = i < xy ? 2 * i + (sel == 2u ? 1 : 0) : 2 * xy + (i - xy);
        const int pos = sel == 3u ? 2 * xy + rest + i : single;
        if (sel) list[pos] = make_entry(kb, sel, valid);
        cx += __popc(bx);
        cy += __popc(by);
        cb += __popc(bb);
      }
      count = nx + ny + cb;
    }
    __syncwarp();
    // leave the byte maps all zero for the next item (16-byte stores; the compaction
    // loops above only read them)
    {
      uint4* z = reinterpret_cast<uint4*>(bm0);
      const int words = (C::kPairs == 2 ? 2 * kMaxNb : kMaxNb) / 16;
      const int used = (nb + 15) / 16;  // words of each map that can hold a 1
      for (int i = (int)lane; i < words; i += 32)
        if ((i % (kMaxNb / 16)) < used) z[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    __syncwarp();
    if (a.n_splits > 1) {
      // this unit's share of the item's key tiles: tiles [t0, t1) of n_t
      const int split = h.item - item * a.n_splits;
      const int n_t = (count + C::kSub - 1) / C::kSub;
      const int t0 = (int)((long long)n_t * split / a.n_splits);
      const int t1 = (int)((long long)n_t * (split + 1) / a.n_splits);
      off = t0 * C::kSub;
      const int end = t1 * C::kSub < count ? t1 * C::kSub : count;
      count = end - off;
    }
  }
  h.count = count;
  if (lane == 0) {
    ctl->hdr_item[buf] = h.item;
    ctl->hdr_n[buf] = count;
    ctl->hdr_off[buf] = off;
    mbar_arrive(&ctl->list_full[buf]);
  }
  __syncwarp();
  return h;
}

// List warp: builds the CTA's work items' lists one item ahead of their use.
template <int BLOCK, bool JENGA>
__device__ void list_role(uint8_t* smem, SmemCtl* ctl, const FwdArgs& a) {
  bool ok = true;
  for (uint32_t it = 0; ok; ++it)
    if (build_list<BLOCK, JENGA>(smem, ctl, a, it, ok).item < 0) break;
}

// TMA warp: Q and the selected K/V tiles of each item, in the order the MMA consumes them.
template <int BLOCK, bool JENGA>
__device__ void tma_role(uint8_t* smem, SmemCtl* ctl, const FwdArgs& a, const CUtensorMap* tq,
                         const CUtensorMap* tk, const CUtensorMap* tv) {
  // one thread issues every copy; its waits are its own (no warp collective follows them)
  using C = Cfg<BLOCK>;
  const uint64_t pol_kv = policy_evict_last();
  const uint64_t pol_q = policy_evict_first();
  uint32_t L = 0;                            // K/V tiles loaded so far (ring position)
  uint32_t qf0 = 0, qf1 = 0;                 // Q copies issued per Q buffer
  bool ok = true;
  for (uint32_t it = 0; ok; ++it) {
    const uint32_t buf = it & 1;
    if (!wait_bar(&ctl->list_full[buf], (it >> 1) & 1, ctl, a, 7)) break;
    const int unit = ctl->hdr_item[buf];
    const int count = ctl->hdr_n[buf];
    if (unit < 0) break;
    const uint32_t* list =
        reinterpret_cast<const uint32_t*>(smem + kOffList) + buf * kMaxNb + ctl->hdr_off[buf];
    const int item = unit / a.n_splits;
    const int bh = item / a.items_per_bh;
    const int qa = (item - bh * a.items_per_bh) * C::kPairs;
    // Q (also the item's output staging buffer): free once the item two back is stored
    if (it >= 2 && !wait_bar(&ctl->q_empty[buf], ((it >> 1) + 1) & 1, ctl, a, 2)) break;
    const int n_tiles = (count + C::kSub - 1) / C::kSub;
    if (n_tiles > 0) {
      // key/value head of this query head (grouped-query attention)
      const int kvh = (bh / a.Hq) * a.Hkv + (bh % a.Hq) / a.group;
      uint8_t* qs = smem + kOffQ + buf * kTileBytes;
      // 128 query rows of head bh; rows past Sq (a lone last block) read as zeros
      mbar_arrive_expect_tx(&ctl->q_full[buf], kTileBytes);
      tma_load_3d_hint(qs, tq, &ctl->q_full[buf], 0, qa * BLOCK, bh, pol_q);
      tma_load_3d_hint(qs + kTileBytes / 2, tq, &ctl->q_full[buf], 64, qa * BLOCK, bh, pol_q);
      if (buf) ++qf1; else ++qf0;
      // K/V tiles in the order the MMA warp consumes them: K0, K1, V0, K2, V1, ...
      for (int t = 0; t <= n_tiles && ok; ++t) {
#pragma unroll
        for (int which = 0; which < 2; ++which) {  // 0: K of tile t, 1: V of tile t-1
          const int tt = which == 0 ? t : t - 1;
          if (tt < 0 || tt >= n_tiles) continue;
          const uint32_t stage = L % kStages;
          if (L >= kStages &&
              !wait_bar(&ctl->kv_empty[stage], ((L / kStages) + 1) & 1, ctl, a, 3)) {
            ok = false;
            break;
          }
          const CUtensorMap* map = which == 0 ? tk : tv;
          uint8_t* dst = smem + kOffKV + stage * kTileBytes;
          const int e0 = tt * C::kSub;
          const int ne = (count - e0) < C::kSub ? (count - e0) : C::kSub;
          mbar_arrive_expect_tx(&ctl->kv_full[stage], (uint32_t)ne * BLOCK * 128 * 2);
          for (int e = 0; e < ne; ++e) {
            const int krow = kvh * a.Sk + (int)(list[e0 + e] & 0xFFFFu) * BLOCK;
            // d-halves are separate [128 rows][64] sub-tiles; block e fills rows e*BLOCK..
            tma_load_2d_hint(dst + e * BLOCK * 128, map, &ctl->kv_full[stage], 0, krow, pol_kv);
            tma_load_2d_hint(dst + kTileBytes / 2 + e * BLOCK * 128, map, &ctl->kv_full[stage],
                             64, krow, pol_kv);
          }
          ++L;
        }
      }
    }
    mbar_arrive(&ctl->list_empty[buf]);  // done reading this item's list
  }
  // drain: every copy this thread issued has landed before the CTA can exit (ring
  // positions 0..L-1 went to stage position % kStages)
  for (uint32_t s = 0; s < (uint32_t)kStages; ++s) {
    const uint32_t fills = L > s ? (L - s + kStages - 1) / kStages : 0;
    if (fills) wait_bar(&ctl->kv_full[s], (fills - 1) & 1, ctl, a, 4, true);
  }
  if (qf0) wait_bar(&ctl->q_full[0], (qf0 - 1) & 1, ctl, a, 5, true);
  if (qf1) wait_bar(&ctl->q_full[1], (qf1 - 1) & 1, ctl, a, 5, true);
}

// ------------------------------------------------------------------------------------
// MMA warp (one thread issues)
// ------------------------------------------------------------------------------------
template <int BLOCK, bool JENGA>
__device__ void mma_role(uint8_t* smem, SmemCtl* ctl, const FwdArgs& a, uint32_t tmem) {
  using C = Cfg<BLOCK>;
  constexpr uint32_t kIdescS128 = idesc_bf16_f32(128, 128, false, false);
  constexpr uint32_t kIdescS64 = idesc_bf16_f32(128, 64, false, false);
  constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 128, false, true);
  uint32_t L = 0;            // ring position
  uint32_t g = 0;            // key tiles issued so far, across items (S buffer g & 1; the
                             // tile's P phase on that buffer is g >> 1)
  uint32_t ne_items = 0;     // non-empty items so far (O phases)
  uint32_t nq0 = 0, nq1 = 0; // Q fills consumed per Q buffer (scalars: no indexed array)
  for (uint32_t it = 0;; ++it) {
    const uint32_t buf = it & 1;
    if (!wait_bar(&ctl->list_full[buf], (it >> 1) & 1, ctl, a, 10)) break;
    const int item = ctl->hdr_item[buf];
    const int count = ctl->hdr_n[buf];
    mbar_arrive(&ctl->list_empty[buf]);
    if (item < 0) break;
    const int n_tiles = (count + C::kSub - 1) / C::kSub;
    if (n_tiles == 0) continue;
    if (!wait_bar(&ctl->q_full[buf], (buf ? nq1 : nq0) & 1, ctl, a, 11)) break;
    if (buf) ++nq1; else ++nq0;
    if (a.stall) {
      // test hook: wait on a barrier no role ever completes, so the wait runs out, the
      // status word records code 31 and every role unwinds (copies already in flight
      // are drained by their issuers)
      wait_bar(&ctl->never, 0, ctl, a, 31);
      break;
    }
    tc_fence_after();
    const uint64_t qdesc = smem_desc_sw128(smem_addr(smem + kOffQ + buf * kTileBytes), 16, 1024);
    bool first[2] = {true, true};  // next PV half w is the item's first into O_w
    bool ok = true;
    for (int t = 0; t <= n_tiles && ok; ++t) {
      if (t < n_tiles) {  // S = Q K_t^T into S buffer (g + t) & 1
        const uint32_t stage = L % kStages;
        if (!wait_bar(&ctl->kv_full[stage], (L / kStages) & 1, ctl, a, 12)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int ne = (count - t * C::kSub) < C::kSub ? (count - t * C::kSub) : C::kSub;
        const uint32_t idesc = (ne * BLOCK == 128) ? kIdescS128 : kIdescS64;
        const uint64_t kdesc =
            smem_desc_sw128(smem_addr(smem + kOffKV + stage * kTileBytes), 16, 1024);
        const uint32_t sb = (g + t) & 1;
        const uint32_t tS = tmem + kColS + sb * 128;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          // the descriptor's start address is addr >> 4 in its low bits: step by offset >> 4
          const uint64_t off16 = ((k >> 2) * (kTileBytes / 2) + (k & 3) * 32) >> 4;
          mma_ss(tS, qdesc + off16, kdesc + off16, idesc, k > 0);
        }
        mma_commit(&ctl->kv_empty[stage]);  // K stage free; S ready
        ++L;
      }
      if (t >= 1) {  // O_w += P V for the previous tile, one key half per warpgroup
        const int tp = t - 1;
        if (tp == 0 && ne_items >= 1 &&
            !wait_bar(&ctl->o_empty, (ne_items - 1) & 1, ctl, a, 13)) {
          ok = false;
          break;
        }
        const uint32_t stage = L % kStages;
        if (!wait_bar(&ctl->kv_full[stage], (L / kStages) & 1, ctl, a, 15)) {
          ok = false;
          break;
        }
        const int ne = (count - tp * C::kSub) < C::kSub ? (count - tp * C::kSub) : C::kSub;
        const int halves = (ne * BLOCK) / 64;  // 1 for a 64-key tile, else 2
        const uint64_t vdesc =
            smem_desc_sw128(smem_addr(smem + kOffKV + stage * kTileBytes), kTileBytes / 2, 1024);
        const uint32_t pb = (g + tp) & 1;
        const uint32_t tS = tmem + kColS + pb * 128;
        bool pw = true;
#pragma unroll
        for (int w = 0; w < 2; ++w) {
          // this half's warpgroup has written its P (both are waited, so every phase of
          // both barriers is consumed, even for a 64-key tile)
          if (!wait_bar(&ctl->p_full[pb * 2 + w], ((g + tp) >> 1) & 1, ctl, a, 14)) {
            pw = false;
            break;
          }
          tc_fence_after();
          if (w >= halves) continue;
          const uint32_t tO = tmem + kColO + w * 128;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            mma_ts(tO, tS + w * 64 + k * 8, vdesc + ((w * 8192 + k * 2048) >> 4), kIdescPV,
                   (!first[w] || k > 0) ? 1u : 0u);
          }
          first[w] = false;
        }
        if (!pw) {
          ok = false;
          break;
        }
        mma_commit(&ctl->kv_empty[stage]);  // V stage free; O holds this tile
        ++L;
      }
    }
    if (!ok) break;
    g += n_tiles;
    mma_commit(&ctl->o_full);
    ++ne_items;
  }
  // every MMA issued has completed before TMEM can be released
  mma_commit(&ctl->drain);
  wait_bar(&ctl->drain, 0, ctl, a, 16, true);
}

// ------------------------------------------------------------------------------------
// softmax warpgroups: thread = query row of the 128-row tile
// ------------------------------------------------------------------------------------
// One key tile for this row: mask, running max, exp2, both row sums, bf16 P written over
// S in TMEM.  l_exact sums the fp32 weights (for lse); l_round sums the bf16-rounded
// weights the PV MMA actually applies (for normalising out), so the weights on V add up
// to one even when the reference max lags the true one.
template <int NK>
__device__ __forceinline__ void softmax_tile(uint32_t tS, int lim0, int lim1, int kps, float sl2,
                                             float& m_run, float& l_exact, float& l_round,
                                             float& alpha) {
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
  float mx[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
  for (int j = 4; j + 1 < NK; j += 8) {
#pragma unroll
    for (int c = 0; c < 4 && j + 2 * c + 1 < NK; ++c)
      mx[c] = fmax3(mx[c], s[j + 2 * c], s[j + 2 * c + 1]);
  }
  const float mraw = fmax3(fmaxf(mx[0], mx[1]), mx[2], mx[3]);
  const float m_tile = mraw * sl2;
  alpha = 1.0f;
  if (m_tile > m_run + kRescaleThreshold) {
    if (m_run != -INFINITY) alpha = fast_exp2(m_run - m_tile);
    m_run = m_tile;
  }
  const float neg = (m_run == -INFINITY) ? 0.0f : -m_run;
  const uint64_t sl2x2 = f32x2(sl2, sl2), negx2 = f32x2(neg, neg);
  uint64_t acc_e[2] = {f32x2(0.f, 0.f), f32x2(0.f, 0.f)};
  float r0 = 0.f, r1 = 0.f, r2 = 0.f, r3 = 0.f;
  uint32_t pk[NK / 2];
#pragma unroll
  for (int i = 0; i < NK / 2; ++i) {
    float y0, y1;
    split_f32x2(fma_f32x2(f32x2(s[2 * i], s[2 * i + 1]), sl2x2, negx2), y0, y1);
    const float p0 = fast_exp2(y0), p1 = fast_exp2(y1);
    acc_e[i & 1] = add_f32x2(acc_e[i & 1], f32x2(p0, p1));
    pk[i] = pack_bf16x2(p0, p1);
    if (i & 1)
      add_bf16x2_to_f32(pk[i], r2, r3);
    else
      add_bf16x2_to_f32(pk[i], r0, r1);
  }
  float e0, e1, e2, e3;
  split_f32x2(acc_e[0], e0, e1);
  split_f32x2(acc_e[1], e2, e3);
  l_exact = l_exact * alpha + ((e0 + e1) + (e2 + e3));
  l_round = l_round * alpha + ((r0 + r1) + (r2 + r3));
#pragma unroll
  for (int c = 0; c < NK / 64; ++c)
    tmem_st_32x32b_x32(tS + c * 32, *reinterpret_cast<const uint32_t(*)[32]>(&pk[c * 32]));
}

template <int BLOCK, bool JENGA>
__device__ void softmax_role(uint8_t* smem, SmemCtl* ctl, const FwdArgs& a, uint32_t tmem,
                             int w, const CUtensorMap* to) {
  using C = Cfg<BLOCK>;
  const int row = threadIdx.x & 127;
  const uint32_t lane_base = (((threadIdx.x >> 5) & 3) * 32) << 16;  // warp's TMEM lanes
  const uint32_t half = (BLOCK == 64) ? (uint32_t)(row >> 6) : 0u;
  const uint32_t tO0 = tmem + kColO + lane_base, tO1 = tO0 + 128;
  const uint32_t tOw = w ? tO1 : tO0;
  float* stats = reinterpret_cast<float*>(smem + kOffStats);  // [par][wg][3][128]
  const bool leader = row == 0;
  uint32_t g = 0;         // key tiles seen so far, across items (S buffer g & 1)
  uint32_t ring = 0;      // ring position of the current item's first K tile
  uint32_t ne_items = 0;
  bool have_prev = false;  // store leader: an item's store whose Q buffer is not yet released
  uint32_t prev_buf = 0;
  for (uint32_t it = 0;; ++it) {
    const uint32_t buf = it & 1;
    if (!wait_warp(&ctl->list_full[buf], (it >> 1) & 1, ctl, a, 20)) break;
    const int unit = ctl->hdr_item[buf];
    const int count = ctl->hdr_n[buf];
    if (unit < 0) break;
    const uint32_t* list =
        reinterpret_cast<const uint32_t*>(smem + kOffList) + buf * kMaxNb + ctl->hdr_off[buf];
    const int item = unit / a.n_splits;
    const int n_tiles = (count + C::kSub - 1) / C::kSub;
    float m_run = -INFINITY, l_exact = 0.0f, l_round = 0.0f;
    bool ok = true;
    bool started = false;  // this warpgroup has a PV in flight for this item
    for (int t = 0; t < n_tiles; ++t, ++g) {
      const int e0 = t * C::kSub;
      const int ne = (count - e0) < C::kSub ? (count - e0) : C::kSub;
      // A 64-key tile has no second half: warpgroup 1 then writes nothing, but still
      // waits for the tile and arrives, so that every phase of both P barriers completes.
      const bool has_half = ne * BLOCK / 64 > w;
      int lim = 0;
      if (has_half) {
        if (BLOCK == 64) {
          lim = entry_limit(list[e0 + w], half);
        } else {
          lim = entry_limit(list[e0], half) - 64 * w;
          lim = lim < 0 ? 0 : (lim > 64 ? 64 : lim);
        }
      }
      const uint32_t sb = g & 1;
      // ring order K0, K1, V0, K2, V1, ...: K(t) sits at t ? 2t - 1 : 0, V(t) at 2t + 2
      const uint32_t kpos = ring + (t ? 2u * t - 1u : 0u);
      if (!wait_warp(&ctl->kv_empty[kpos % kStages], (kpos / kStages) & 1, ctl, a, 21)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t tS = tmem + kColS + sb * 128 + 64 * w + lane_base;
      float alpha = 1.0f;
      if (lim > 0) {
        softmax_tile<64>(tS, lim, 64, 64, a.scale_log2, m_run, l_exact, l_round, alpha);
      } else if (has_half) {
        // none of this warp's rows attends these keys (a block selected only by the other
        // query block of the pair, or a zero-width tail): P = 0, the running state stays.
        // lim depends only on the row's query half, so the branch is warp-uniform.
        uint32_t z[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) z[j] = 0u;
        tmem_st_32x32b_x32(tS, z);
      }
      // O rescale when this row's reference max moved: wait until the previous tile's PV
      // has completed (TMEM access is warp-collective, hence the vote).
      if (__any_sync(0xffffffffu, alpha != 1.0f) && started) {
        const uint32_t vpos = ring + 2u * t;  // V(t - 1)
        if (!wait_warp(&ctl->kv_empty[vpos % kStages], (vpos / kStages) & 1, ctl, a, 25)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(tOw + c * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
          tmem_st_32x32b_x32(tOw + c * 32, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if ((threadIdx.x & 31) == 0) mbar_arrive(&ctl->p_full[sb * 2 + w]);
      started = true;
      if (leader && have_prev) {  // the previous item's store has had a tile to read
        bulk_wait_group_read0();
        mbar_arrive(&ctl->q_empty[prev_buf]);
        have_prev = false;
      }
    }
    if (!ok) break;
    ring += 2u * (uint32_t)n_tiles;  // the item's K and V tiles
    // ---- merge the two halves of the key walk, then this warpgroup's half of the output
    float* st = stats + buf * (2 * 3 * 128);
    st[(w * 3 + 0) * 128 + row] = m_run;
    st[(w * 3 + 1) * 128 + row] = l_exact;
    st[(w * 3 + 2) * 128 + row] = l_round;
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&ctl->stats_bar[buf]);
    if (n_tiles > 0) {
      if (!wait_warp(&ctl->o_full, ne_items & 1, ctl, a, 22)) break;
      tc_fence_after();
    }
    if (!wait_warp(&ctl->stats_bar[buf], (it >> 1) & 1, ctl, a, 23)) break;
    float m[2], le[2], lr[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      m[h] = st[(h * 3 + 0) * 128 + row];
      le[h] = st[(h * 3 + 1) * 128 + row];
      lr[h] = st[(h * 3 + 2) * 128 + row];
    }
    const float mm = fmaxf(m[0], m[1]);
    float c[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) c[h] = lr[h] > 0.0f ? fast_exp2(m[h] - mm) : 0.0f;
    const float l_r = c[0] * lr[0] + c[1] * lr[1];
    const float l_e = c[0] * le[0] + c[1] * le[1];
    const bool has = l_r > 0.0f;
    const float inv = has ? 1.0f / l_r : 0.0f;
    // split-KV units keep O unnormalised (relative to mm): the merge kernel divides
    const bool split = a.part != nullptr;
    float* part = split ? a.part + (size_t)unit * kPartFloats : nullptr;
    const float f0 = split ? c[0] : c[0] * inv, f1 = split ? c[1] : c[1] * inv;
    // a half's O is read only if that half attended something in this item (the other
    // accumulator may still hold an earlier item's values)
    const bool use0 = __any_sync(0xffffffffu, lr[0] > 0.0f);
    const bool use1 = __any_sync(0xffffffffu, lr[1] > 0.0f);
    const int bh = item / a.items_per_bh;
    const int qa = (item - bh * a.items_per_bh) * C::kPairs;
    uint8_t* qs = smem + kOffQ + buf * kTileBytes + w * (kTileBytes / 2);
#pragma unroll 1
    for (int cc = 0; cc < 4; ++cc) {  // this warpgroup's 64 output columns, 16 at a time
      const uint32_t col = w * 64 + cc * 16;
      uint32_t o0[16], o1[16];
      if (use0) tmem_ld_32x32b_x16(tO0 + col, o0);
      if (use1) tmem_ld_32x32b_x16(tO1 + col, o1);
      tmem_wait_ld();
      float x[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        float v = 0.0f;
        if (use0 && f0 != 0.0f) v = __uint_as_float(o0[k]) * f0;
        if (use1 && f1 != 0.0f) v = fmaf(__uint_as_float(o1[k]), f1, v);
        x[k] = v;
      }
      if (split) {
        float4* dst = reinterpret_cast<float4*>(part + row * 128 + col);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          dst[j] = make_float4(x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]);
        continue;
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        uint32_t wv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) wv[j] = pack_bf16x2(x[8 * i + 2 * j], x[8 * i + 2 * j + 1]);
        const uint32_t chunk = (uint32_t)(cc * 2 + i);      // 16-byte chunk in the 128B row
        const uint32_t phys = chunk ^ (uint32_t)(row & 7);  // 128-byte swizzle
        uint8_t* dst = qs + row * 128 + phys * 16;
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(smem_addr(dst)), "r"(wv[0]),
                     "r"(wv[1]), "r"(wv[2]), "r"(wv[3])
                     : "memory");
      }
    }
    if (split) {
      if (w == 0) {
        part[128 * 128 + row] = has ? mm : -INFINITY;
        part[128 * 128 + 128 + row] = l_r;
        part[128 * 128 + 256 + row] = l_e;
      }
    } else if (w == 0 && a.lse != nullptr && qa * BLOCK + row < a.Sq) {
      a.lse[(long long)bh * a.Sq + qa * BLOCK + row] = has ? mm + log2f(l_e) : -3.402823466e+38f;
    }
    tc_fence_before();
    fence_proxy_async_smem();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) {
      if (n_tiles > 0) mbar_arrive(&ctl->o_empty);
      mbar_arrive(&ctl->list_empty[buf]);
      mbar_arrive(&ctl->epi_bar[w]);
    }
    if (n_tiles > 0) ++ne_items;
    // the leader waits alone; the vote keeps the decision to stop warp-uniform
    const bool stored = !leader || wait_bar(&ctl->epi_bar[w], it & 1, ctl, a, 24);
    if (!__all_sync(0xffffffffu, stored)) break;
    if (leader) {
      if (have_prev) {  // an item without tiles in between: release the older buffer now
        bulk_wait_group_read0();
        mbar_arrive(&ctl->q_empty[prev_buf]);
      }
      if (!split) {
        tma_store_3d(to, qs, w * 64, qa * BLOCK, bh);  // rows past Sq are not written
        bulk_commit_group();
      }
      have_prev = true;
      prev_buf = buf;
    }
  }
  if (leader) {
    bulk_wait_group0();
    if (have_prev) mbar_arrive(&ctl->q_empty[prev_buf]);
  }
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
      mbar_init(&ctl->list_full[i], 1);
      mbar_init(&ctl->list_empty[i], 10);  // the TMA warp, the MMA thread, 8 softmax warps
      mbar_init(&ctl->q_full[i], 1);
      mbar_init(&ctl->q_empty[i], 2);     // one TMA-store leader per softmax warpgroup
      mbar_init(&ctl->p_full[i], 4);
      mbar_init(&ctl->p_full[i + 2], 4);
      mbar_init(&ctl->stats_bar[i], 8);
      mbar_init(&ctl->epi_bar[i], 4);
    }
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&ctl->kv_full[i], 1);
      mbar_init(&ctl->kv_empty[i], 1);
    }
    mbar_init(&ctl->o_full, 1);
    mbar_init(&ctl->o_empty, 8);
    mbar_init(&ctl->drain, 1);
    mbar_init(&ctl->vbs_ready, 1);
    mbar_init(&ctl->never, 1);
    ctl->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 8) {
    // the byte maps start (and are always left) all zero
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

  if (warp < 8) {
    regs_increase<kSoftmaxRegs>();
    softmax_role<BLOCK, JENGA>(smem, ctl, a, tmem, (int)(warp >> 2), &to);
  } else {
    regs_decrease<kOtherRegs>();
    if (warp == 8) {
      if (lane_id() == 0) tma_role<BLOCK, JENGA>(smem, ctl, a, &tq, &tk, &tv);
      __syncwarp();
    } else if (warp == 10) {
      list_role<BLOCK, JENGA>(smem, ctl, a);
    } else if (warp == 9) {
      if (lane_id() == 0) mma_role<BLOCK, JENGA>(smem, ctl, a, tmem);
      __syncwarp();
    } else if (warp == 11 && a.vbs != nullptr) {
      // variable_block_sizes, clamped, into SMEM once per CTA, while the list warp loads
      // the first item's LUT rows: the compaction reads one entry per selected block, and
      // from global memory each would cost a round trip of its own
      const uint32_t lane = lane_id();
      uint8_t* vt = smem + kOffVbs;
      for (int base = 0; base < a.nbk; base += 32 * 16) {
        int v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int kb = base + 32 * j + (int)lane;
          v[j] = kb < a.nbk ? __ldg(a.vbs + kb) : 0;
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int kb = base + 32 * j + (int)lane;
          if (kb < a.nbk) vt[kb] = (uint8_t)(v[j] < 0 ? 0 : (v[j] > BLOCK ? BLOCK : v[j]));
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->vbs_ready);
    }
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

// ------------------------------------------------------------------------------------
// Split-KV merge: one warp per query row combines the row's n_splits partials exactly as
// the forward merges its two key halves: M = max m_s, c_s = 2^(m_s - M) (0 for an empty
// partial), out = sum c_s O_s / sum c_s l_round_s, lse = M + log2(sum c_s l_exact_s).
// Partials of item i are units i * n_splits .. i * n_splits + n_splits - 1.
template <int BLOCK>
__global__ void __launch_bounds__(256) split_merge_kernel(const float* __restrict__ part,
                                                          int n_items, int n_splits,
                                                          int items_per_bh, int Sq,
                                                          uint16_t* __restrict__ out,
                                                          float* __restrict__ lse) {
  using C = Cfg<BLOCK>;
  const long long r = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);  // item * 128 + row
  if (r >= (long long)n_items * 128) return;
  const int item = (int)(r >> 7), row = (int)(r & 127);
  const int bh = item / items_per_bh;
  const int qrow = (item - bh * items_per_bh) * C::kPairs * BLOCK + row;
  if (qrow >= Sq) return;  // the rows past a lone last query block
  const uint32_t lane = threadIdx.x & 31;
  const float* p0 = part + (size_t)item * n_splits * kPartFloats;
  // the row's statistics of splits lane and lane + 32 (n_splits <= 64), read in parallel
  float m[2], l_r[2], l_e[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int s = (int)lane + 32 * h;
    m[h] = -INFINITY;
    l_r[h] = 0.0f;
    l_e[h] = 0.0f;
    if (s < n_splits) {
      const float* st = p0 + (size_t)s * kPartFloats + 128 * 128;
      m[h] = st[row];
      l_r[h] = st[128 + row];
      l_e[h] = st[256 + row];
    }
  }
  float M = -INFINITY;
#pragma unroll
  for (int h = 0; h < 2; ++h)
    if (l_r[h] > 0.0f) M = fmaxf(M, m[h]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float c[2], lr = 0.0f, le = 0.0f;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    c[h] = l_r[h] > 0.0f ? exp2f(m[h] - M) : 0.0f;
    lr = fmaf(c[h], l_r[h], lr);
    le = fmaf(c[h], l_e[h], le);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lr += __shfl_xor_sync(0xffffffffu, lr, o);
    le += __shfl_xor_sync(0xffffffffu, le, o);
  }
  // O: this lane's 4 columns of each split's partial, four splits' loads at a time, summed
  // in split order
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < n_splits; s0 += 4) {
    float cs[4];
    float4 o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int s = s0 + j;
      const float cj = __shfl_sync(0xffffffffu, (s & 32) ? c[1] : c[0], s & 31);
      cs[j] = s < n_splits ? cj : 0.0f;
      o[j] = cs[j] != 0.0f
                 ? reinterpret_cast<const float4*>(p0 + (size_t)s * kPartFloats + row * 128)[lane]
                 : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      acc.x = fmaf(cs[j], o[j].x, acc.x);
      acc.y = fmaf(cs[j], o[j].y, acc.y);
      acc.z = fmaf(cs[j], o[j].z, acc.z);
      acc.w = fmaf(cs[j], o[j].w, acc.w);
    }
  }
  const bool has = lr > 0.0f;
  const float inv = has ? 1.0f / lr : 0.0f;
  const long long orow = (long long)bh * Sq + qrow;
  uint2 packed;
  packed.x = pack_bf16x2(has ? acc.x * inv : 0.0f, has ? acc.y * inv : 0.0f);
  packed.y = pack_bf16x2(has ? acc.z * inv : 0.0f, has ? acc.w * inv : 0.0f);
  reinterpret_cast<uint2*>(out + orow * 128)[lane] = packed;
  if (lse != nullptr && lane == 0) lse[orow] = has ? M + log2f(le) : -3.402823466e+38f;
}

}  // namespace vsa
