// vsa_api.cu -- the C ABI of libvsa_gb300.so (declared in include/vsa.h): host-side
// argument checks, TMA tensor-map encoding, persistent-grid launches of the forward
// (LUT, block-map, grouped-query, cross-length and split-KV routes) and of the backward,
// the metadata conversion kernels, the host-buffer wrapper and the device status word.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/vsa.h"
#include "vsa_fwd_kernel.cuh"
#include "vsa_bwd_kernel.cuh"

namespace vsa {

// Device status word: a kernel that gives up on a bounded wait records a code here.
__device__ unsigned int g_status = 0;

// ------------------------------------------------------------------ metadata kernels
// LUT -> bitmap.  One CTA per row: zero the row, then scatter 1 at every listed block.
__global__ void lut_to_bitmap_kernel(const int32_t* __restrict__ idx,
                                     const int32_t* __restrict__ num, int max_kv, int nb,
                                     int8_t* __restrict__ bitmap) {
  const long long r = blockIdx.x;
  int8_t* row = bitmap + r * nb;
  for (int kb = threadIdx.x; kb < nb; kb += blockDim.x) row[kb] = 0;
  __syncthreads();
  int n = num[r];
  n = n < 0 ? 0 : (n > max_kv ? max_kv : n);
  const int32_t* lut = idx + r * max_kv;
  for (int s = threadIdx.x; s < n; s += blockDim.x) {
    const int kb = lut[s];
    if (kb >= 0 && kb < nb) row[kb] = 1;
  }
}

// bitmap -> LUT.  One warp per row: ascending ballot/popc compaction, then -1 padding.
__global__ void bitmap_to_lut_kernel(const int8_t* __restrict__ bitmap, int rows, int nb,
                                     int max_kv, int32_t* __restrict__ idx,
                                     int32_t* __restrict__ num) {
  const long long r = (long long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x / 32);
  if (r >= rows) return;
  const unsigned lane = threadIdx.x & 31;
  const int8_t* row = bitmap + r * nb;
  int32_t* out = idx + r * max_kv;
  int count = 0;
  for (int base = 0; base < nb && count < max_kv; base += 32) {
    const int kb = base + (int)lane;
    const bool sel = kb < nb && row[kb] != 0;
    const unsigned ballot = __ballot_sync(0xffffffffu, sel);
    const int pos = count + __popc(ballot & ((1u << lane) - 1u));
    if (sel && pos < max_kv) out[pos] = kb;
    count += __popc(ballot);
  }
  if (count > max_kv) count = max_kv;
  for (int s = count + (int)lane; s < max_kv; s += 32) out[s] = -1;
  if (lane == 0) num[r] = count;
}

}  // namespace vsa

using namespace vsa;

namespace {

thread_local int t_last_launches = 0;

// Timeout-path test hooks (vsa_set_wait_limit_ns, vsa_set_stall_test), read at launch.
std::atomic<unsigned long long> g_wait_ns{0};  // 0 = the kernels' full limit
std::atomic<int> g_stall{0};

unsigned long long launch_wait_ns(uint64_t full) {
  const unsigned long long ns = g_wait_ns.load();
  return ns == 0 ? full : ns;
}

struct DeviceInfo {
  bool ready = false;
  int sm_count = 0;
  int major = 0, minor = 0;
  bool attr_set[4] = {false, false, false, false};
  int regs[4] = {0, 0, 0, 0};
  bool bwd_attr_set[2] = {false, false};
};
std::mutex g_mu;
DeviceInfo g_dev[64];

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

vsa_status device_info(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return VSA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return VSA_ERR_CUDA;
    d.ready = true;
  }
  *out = &d;
  return VSA_OK;
}

// 2-D view [rows, 128] of a BHSD bf16 tensor, 128-byte swizzle, box {64, box_rows}.
bool make_map(CUtensorMap* m, const void* ptr, long long rows, int box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {128, (cuuint64_t)rows};
  cuuint64_t strides[1] = {128 * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D view [heads, seq, 128] of a BHSD bf16 tensor, box {64, box_rows, 1}: a box that runs
// past the end of a head's sequence is clipped there (loads read zeros, stores drop the
// rows) instead of spilling into the next head.
bool make_map_3d(CUtensorMap* m, const void* ptr, long long heads, long long seq,
                 int box_rows = 128) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {128, (cuuint64_t)seq, (cuuint64_t)heads};
  cuuint64_t strides[2] = {128 * 2, (cuuint64_t)seq * 128 * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb_) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb_ && y < x + na;
}

// Problem shape shared by every forward entry point: q / out [B, Hq, Sq, D],
// k / v [B, Hkv, Sk, D], lse [B, Hq, Sq].
struct Shape {
  int B, Hq, Hkv, Sq, Sk, D, block;
  float scale;
  long long rows_q() const { return (long long)B * Hq * Sq; }
  long long rows_k() const { return (long long)B * Hkv * Sk; }
};

// Host-side checks of a forward call (no device reads).  `nothing` is set when there is
// no output row to write.
vsa_status check_shape(const void* q, const void* k, const void* v, const void* out,
                       const float* lse, const Shape& p, DeviceInfo** dev, bool* nothing) {
  *nothing = false;
  if (p.B < 0 || p.Hq < 0 || p.Hkv < 0 || p.Sq < 0 || p.Sk < 0) return VSA_ERR_INVALID_ARG;
  if (p.D != VSA_HEAD_DIM) return VSA_ERR_UNSUPPORTED;
  if (p.block != 64 && p.block != 128) return VSA_ERR_UNSUPPORTED;
  if (!(p.scale > 0.0f) || !std::isfinite(p.scale)) return VSA_ERR_INVALID_ARG;
  if (p.Sq % p.block != 0 || p.Sk % p.block != 0) return VSA_ERR_INVALID_ARG;
  if (p.Hq > 0 && (p.Hkv < 1 || p.Hq % p.Hkv != 0)) return VSA_ERR_INVALID_ARG;
  if (p.Sk / p.block > VSA_MAX_BLOCKS) return VSA_ERR_UNSUPPORTED;
  if (p.rows_q() > (long long)INT_MAX || p.rows_k() > (long long)INT_MAX)
    return VSA_ERR_UNSUPPORTED;
  if (p.rows_q() == 0) {
    *nothing = true;
    return VSA_OK;
  }
  const bool keys = p.rows_k() > 0;
  if (!q || !out || (keys && (!k || !v))) return VSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out) || (keys && (!aligned16(k) || !aligned16(v))))
    return VSA_ERR_INVALID_ARG;
  const size_t qbytes = (size_t)p.rows_q() * p.D * 2, kbytes = (size_t)p.rows_k() * p.D * 2;
  if (overlaps(out, qbytes, q, qbytes) ||
      (keys && (overlaps(out, qbytes, k, kbytes) || overlaps(out, qbytes, v, kbytes))))
    return VSA_ERR_INVALID_ARG;
  if (lse && overlaps(lse, (size_t)p.rows_q() * 4, out, qbytes)) return VSA_ERR_INVALID_ARG;
  vsa_status st = device_info(dev);
  if (st != VSA_OK) return st;
  if ((*dev)->major != 10 || (*dev)->minor != 3) return VSA_ERR_UNSUPPORTED;
  return VSA_OK;
}

// FwdArgs fields that follow from the shape alone.
FwdArgs shape_args(const Shape& p, float* lse, void* workspace, unsigned int* status) {
  FwdArgs a{};
  a.lse = lse;
  a.sched = static_cast<unsigned int*>(workspace);
  a.status = status;
  a.Hq = p.Hq;
  a.Hkv = p.Hkv;
  a.group = p.Hq / p.Hkv;
  a.Sq = p.Sq;
  a.Sk = p.Sk;
  a.nbq = p.Sq / p.block;
  a.nbk = p.Sk / p.block;
  a.items_per_bh = p.block == 64 ? (a.nbq + 1) / 2 : a.nbq;
  a.n_items = (int)((long long)p.B * p.Hq * a.items_per_bh);
  a.n_splits = 1;
  a.part = nullptr;
  a.scale_log2 = p.scale * 1.4426950408889634f;
  a.wait_ns = launch_wait_ns(kWaitLimitNs);
  a.stall = g_stall.load();
  return a;
}

// One-time per-device kernel attributes (dynamic SMEM limit, registers at launch) and the
// register-pool check; enqueues nothing.
template <int BLOCK, bool JENGA>
vsa_status prepare_fwd(DeviceInfo* dev, int slot) {
  auto kern = bsa_fwd_kernel<BLOCK, JENGA>;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!dev->attr_set[slot]) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kSmemBytes) != cudaSuccess)
        return VSA_ERR_CUDA;
      cudaFuncAttributes fa;
      if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return VSA_ERR_CUDA;
      dev->regs[slot] = fa.numRegs;
      dev->attr_set[slot] = true;
    }
  }
  // The kernel moves registers between warpgroups (setmaxnreg); the launch must provide
  // the pool that re-balancing draws on, or a warpgroup would wait for registers forever.
  if ((long long)dev->regs[slot] * kThreads < (long long)kRegPoolNeeded) return VSA_ERR_UNSUPPORTED;
  return VSA_OK;
}

template <int BLOCK, bool JENGA>
vsa_status launch_fwd(DeviceInfo* dev, int slot, const void* q, const void* k, const void* v,
                      void* out, const Shape& p, const FwdArgs& args, cudaStream_t stream) {
  auto kern = bsa_fwd_kernel<BLOCK, JENGA>;
  vsa_status st = prepare_fwd<BLOCK, JENGA>(dev, slot);
  if (st != VSA_OK) return st;
  // With no keys at all (Sk == 0) no K/V copy is ever issued; the maps only need to encode.
  const bool keys = p.rows_k() > 0;
  const void* kp = keys ? k : q;
  const void* vp = keys ? v : q;
  const long long krows = keys ? p.rows_k() : p.rows_q();
  CUtensorMap tq, tk, tv, to;
  if (!make_map_3d(&tq, q, (long long)p.B * p.Hq, p.Sq) || !make_map(&tk, kp, krows, BLOCK) ||
      !make_map(&tv, vp, krows, BLOCK) || !make_map_3d(&to, out, (long long)p.B * p.Hq, p.Sq))
    return VSA_ERR_CUDA;
  // one CTA per work item up to one per SM (a launch with fewer items than SMs -- the
  // split-KV decode shape -- runs every item at once: 24 heads x 6 ranges of 98,304 keys
  // measured 88 us against 105 us with two items per CTA)
  const int ctas = args.n_items;
  const int grid = ctas < dev->sm_count ? ctas : dev->sm_count;
  kern<<<grid, kThreads, kSmemBytes, stream>>>(tq, tk, tv, to, args);
  if (cudaGetLastError() != cudaSuccess) return VSA_ERR_CUDA;
  t_last_launches = 1;
  if (args.n_splits > 1) {
    const int items = args.n_items / args.n_splits;
    const long long rows = (long long)items * 128;
    split_merge_kernel<BLOCK><<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(
        args.part, items, args.n_splits, args.items_per_bh, args.Sq,
        static_cast<uint16_t*>(out), args.lse);
    if (cudaGetLastError() != cudaSuccess) return VSA_ERR_CUDA;
    t_last_launches = 2;
  }
  return VSA_OK;
}

unsigned int* status_word() {
  unsigned int* status = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&status), g_status) != cudaSuccess)
    return nullptr;
  return status;
}

// the scheduling counters at the start of a workspace
constexpr size_t kSchedBytes = 256;

bool workspace_ok(const void* workspace) {
  return workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 3u) == 0;
}

// LUT-driven forward (VSA), any head grouping and lengths.
vsa_status run_lut(const vsa_bf16* q, const vsa_bf16* k, const vsa_bf16* v,
                   const int32_t* q2k_idx, const int32_t* q2k_num, const int32_t* vbs,
                   const Shape& p, int max_kv, vsa_bf16* out, float* lse, void* workspace,
                   vsa_stream_t stream, bool require_vbs, int n_splits = 1,
                   size_t workspace_bytes = 0) {
  t_last_launches = 0;
  DeviceInfo* dev = nullptr;
  bool nothing = false;
  vsa_status st = check_shape(q, k, v, out, lse, p, &dev, &nothing);
  if (st != VSA_OK || nothing) return st;
  if (max_kv < 1) return VSA_ERR_INVALID_ARG;
  if (!q2k_idx || !q2k_num || (require_vbs && !vbs)) return VSA_ERR_INVALID_ARG;
  if (!workspace_ok(workspace)) return VSA_ERR_INVALID_ARG;
  unsigned int* status = status_word();
  if (status == nullptr) return VSA_ERR_CUDA;
  FwdArgs a = shape_args(p, lse, workspace, status);
  a.q2k_idx = q2k_idx;
  a.q2k_num = q2k_num;
  a.vbs = vbs;
  a.max_kv = max_kv;
  if (n_splits > 1) {
    // units (item, key-tile range); partials after the scheduling counters
    const long long units = (long long)a.n_items * n_splits;
    if (units > (long long)INT_MAX) return VSA_ERR_UNSUPPORTED;
    const size_t need = kSchedBytes + (size_t)units * kPartFloats * sizeof(float);
    if (workspace == nullptr || workspace_bytes < need ||
        (reinterpret_cast<uintptr_t>(workspace) & 15u))
      return VSA_ERR_INVALID_ARG;
    const size_t qbytes = (size_t)p.rows_q() * p.D * 2;
    if (overlaps(workspace, need, out, qbytes) || (lse && overlaps(workspace, need, lse,
                                                                    (size_t)p.rows_q() * 4)) ||
        overlaps(workspace, need, q, qbytes))
      return VSA_ERR_INVALID_ARG;
    a.n_splits = n_splits;
    a.n_items = (int)units;
    a.part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + kSchedBytes);
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (p.block == 64) return launch_fwd<64, false>(dev, 0, q, k, v, out, p, a, s);
  return launch_fwd<128, false>(dev, 1, q, k, v, out, p, a, s);
}

// Block-map-driven forward: one int8 map per (b, hq) (bh_stride = nbq * nbk) or one map
// shared by all of them (bh_stride = 0); the kernel compacts each map row itself.
vsa_status run_map(const vsa_bf16* q, const vsa_bf16* k, const vsa_bf16* v,
                   const int8_t* block_map, long long bh_stride, const int32_t* vbs,
                   const Shape& p, vsa_bf16* out, float* lse, void* workspace,
                   vsa_stream_t stream) {
  t_last_launches = 0;
  DeviceInfo* dev = nullptr;
  bool nothing = false;
  vsa_status st = check_shape(q, k, v, out, lse, p, &dev, &nothing);
  if (st != VSA_OK || nothing) return st;
  if (!block_map) return VSA_ERR_INVALID_ARG;
  if (!workspace_ok(workspace)) return VSA_ERR_INVALID_ARG;
  unsigned int* status = status_word();
  if (status == nullptr) return VSA_ERR_CUDA;
  FwdArgs a = shape_args(p, lse, workspace, status);
  a.bitmap = block_map;
  a.bitmap_bh_stride = bh_stride;
  a.vbs = vbs;
  a.max_kv = 1;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (p.block == 64) return launch_fwd<64, true>(dev, 2, q, k, v, out, p, a, s);
  return launch_fwd<128, true>(dev, 3, q, k, v, out, p, a, s);
}

// Limits of the backward's step list (an entry packs the query block in 16 bits and the
// query head within the key/value group in 12 bits).
constexpr long long kBwdMaxQBlocks = 65536, kBwdMaxGroup = 4096;

size_t align256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }

// Backward workspace: the 0/1 block map, D per query row, the fp32 dQ accumulator.
struct BwdLayout {
  size_t bitmap, dvec, dq, total;
};
BwdLayout bwd_layout(long long B, long long Hq, long long Sq, long long Sk, int block) {
  const long long nbq = Sq / block, nbk = Sk / block, rows = B * Hq * Sq;
  BwdLayout l;
  l.bitmap = 0;
  l.dvec = align256((size_t)(B * Hq * nbq * nbk));
  l.dq = l.dvec + align256((size_t)rows * 8);  // -D, then -lse
  l.total = l.dq + (size_t)rows * 128 * 4;
  return l;
}

// The backward: one CTA per key tile of 128 keys (a key block, or an adjacent pair of
// block-64 key blocks).
template <int BLOCK>
vsa_status launch_bwd(DeviceInfo* dev, const BwdArgs& a, const void* q, const void* k,
                      const void* v, const void* dout, long long rows_q, long long kv_heads,
                      long long n_ctas, cudaStream_t s) {
  auto kern = bwd::bsa_bwd_kernel<BLOCK>;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!dev->bwd_attr_set[BLOCK == 128]) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)bwd::kSmemBytes) != cudaSuccess)
        return VSA_ERR_CUDA;
      dev->bwd_attr_set[BLOCK == 128] = true;
    }
  }
  if (n_ctas == 0) return VSA_OK;
  // Q and dO: [rows, 128] with 64-row boxes (a step); K and V: [heads, Sk, 128] with
  // 128-row boxes (a key tile; the rows of a lone last block-64 key block past the end of
  // a head read as zeros)
  CUtensorMap tq, tdo, tk, tv;
  if (!make_map(&tq, q, rows_q, 64) || !make_map(&tdo, dout, rows_q, 64) ||
      !make_map_3d(&tk, k, kv_heads, a.Sk) || !make_map_3d(&tv, v, kv_heads, a.Sk))
    return VSA_ERR_CUDA;
  kern<<<(unsigned)n_ctas, bwd::kThreads, bwd::kSmemBytes, s>>>(tq, tdo, tk, tv, a);
  return cudaGetLastError() == cudaSuccess ? VSA_OK : VSA_ERR_CUDA;
}

// Streams and events of vsa_fwd_from_host, created once per device (no device memory).
// vsa_fwd_from_host: chunks of about kHostChunkBytes of q, k, v each (at most kHostChunks,
// at most one per head).  Measured on GB300 (pinned copies ~210 GB/s one way, ~335 GB/s
// both ways at once): 24 one-head chunks on B1 H24 S98304 ran 4 % faster end to end than
// 8, while on B1 H12 S16384 12 chunks ran 14 % slower than 8 and 4 chunks 4 % slower.
constexpr int kHostChunks = 32;
constexpr size_t kHostChunkBytes = (size_t)20 << 20;
struct HostPipe {
  bool ready = false;
  std::mutex mu;  // one host-buffer call at a time enqueues on these streams
  cudaStream_t s_in = nullptr, s_out = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr, ev_join_in = nullptr;
  cudaEvent_t ev_in[kHostChunks] = {}, ev_done[kHostChunks] = {};
};
HostPipe g_pipe[64];

vsa_status host_pipe(HostPipe** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return VSA_ERR_CUDA;
  HostPipe& p = g_pipe[dev];
  std::lock_guard<std::mutex> lk(g_mu);
  if (!p.ready) {
    const unsigned ev = cudaEventDisableTiming;
    if (cudaStreamCreateWithFlags(&p.s_in, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&p.s_out, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.ev_fork, ev) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.ev_join, ev) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.ev_join_in, ev) != cudaSuccess)
      return VSA_ERR_CUDA;
    for (int c = 0; c < kHostChunks; ++c)
      if (cudaEventCreateWithFlags(&p.ev_in[c], ev) != cudaSuccess ||
          cudaEventCreateWithFlags(&p.ev_done[c], ev) != cudaSuccess)
        return VSA_ERR_CUDA;
    p.ready = true;
  }
  *out = &p;
  return VSA_OK;
}

}  // namespace

extern "C" {

size_t vsa_workspace_bytes(void) { return kSchedBytes; }

size_t vsa_bwd_workspace_bytes(int B, int Hq, int Sq, int Sk, int block) {
  if (B < 0 || Hq < 0 || Sq < 0 || Sk < 0 || (block != 64 && block != 128) ||
      Sq % block != 0 || Sk % block != 0 || Sq / block > kBwdMaxQBlocks)
    return 0;
  return bwd_layout(B, Hq, Sq, Sk, block).total;
}

vsa_status vsa_bwd(const vsa_bf16* q, const vsa_bf16* k, const vsa_bf16* v,
                   const vsa_bf16* out, const vsa_bf16* dout, const float* lse,
                   const int32_t* q2k_idx, const int32_t* q2k_num,
                   const int32_t* variable_block_sizes, int B, int Hq, int Hkv, int Sq, int Sk,
                   int D, int max_kv, int block, float scale, vsa_bf16* dq, vsa_bf16* dk,
                   vsa_bf16* dv, void* workspace, size_t workspace_bytes,
                   vsa_stream_t stream) {
  t_last_launches = 0;
  if ((block == 64 || block == 128) &&
      ((long long)Sq / block > kBwdMaxQBlocks || (Hkv > 0 && Hq / Hkv > kBwdMaxGroup)))
    return VSA_ERR_UNSUPPORTED;
  const Shape p{B, Hq, Hkv, Sq, Sk, D, block, scale};
  DeviceInfo* dev = nullptr;
  bool nothing = false;
  // the forward's checks on q, k, v and out (out is read here, never written)
  vsa_status st = check_shape(q, k, v, out, lse, p, &dev, &nothing);
  if (st != VSA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t kbytes = (size_t)p.rows_k() * 128 * 2, qbytes = (size_t)p.rows_q() * 128 * 2;
  if (nothing) {  // no query rows: every key gets a zero gradient
    if (p.rows_k() == 0) return VSA_OK;
    if (!dk || !dv) return VSA_ERR_INVALID_ARG;
    if (cudaMemsetAsync(dk, 0, kbytes, s) != cudaSuccess ||
        cudaMemsetAsync(dv, 0, kbytes, s) != cudaSuccess)
      return VSA_ERR_CUDA;
    return VSA_OK;
  }
  if (max_kv < 1 || !q2k_idx || !q2k_num || !dout || !lse || !dq) return VSA_ERR_INVALID_ARG;
  if (p.rows_k() > 0 && (!dk || !dv)) return VSA_ERR_INVALID_ARG;
  if (!aligned16(dout) || !aligned16(dq) || !aligned16(lse) ||
      (p.rows_k() > 0 && (!aligned16(dk) || !aligned16(dv))))
    return VSA_ERR_INVALID_ARG;
  const BwdLayout lay = bwd_layout(B, Hq, Sq, Sk, block);
  if (!workspace || workspace_bytes < lay.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return VSA_ERR_INVALID_ARG;
  // outputs must not overlap any input or one another
  const void* ins[6] = {q, k, v, out, dout, lse};
  const size_t insz[6] = {qbytes, kbytes, kbytes, qbytes, qbytes, (size_t)p.rows_q() * 4};
  const void* outs[4] = {dq, dk, dv, workspace};
  const size_t outsz[4] = {qbytes, kbytes, kbytes, lay.total};
  for (int o = 0; o < 4; ++o) {
    for (int i = 0; i < 6; ++i)
      if (outsz[o] && insz[i] && outs[o] && ins[i] && overlaps(outs[o], outsz[o], ins[i], insz[i]))
        return VSA_ERR_INVALID_ARG;
    for (int o2 = o + 1; o2 < 4; ++o2)
      if (outsz[o] && outsz[o2] && outs[o] && outs[o2] &&
          overlaps(outs[o], outsz[o], outs[o2], outsz[o2]))
        return VSA_ERR_INVALID_ARG;
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int8_t* bitmap = reinterpret_cast<int8_t*>(ws + lay.bitmap);
  float* dq_acc = reinterpret_cast<float*>(ws + lay.dq);
  const int nbq = Sq / block, nbk = Sk / block;
  const long long lut_rows = (long long)B * Hq * nbq, rows = p.rows_q();
  float* nD = reinterpret_cast<float*>(ws + lay.dvec);
  float* nlse = nD + rows;
  int launches = 0;
  if (nbk > 0) {
    lut_to_bitmap_kernel<<<(unsigned)lut_rows, 128, 0, s>>>(q2k_idx, q2k_num, max_kv, nbk,
                                                            bitmap);
    ++launches;
  }
  bwd_prep_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(out, dout, lse, rows, nD, nlse);
  ++launches;
  if (cudaGetLastError() != cudaSuccess ||
      cudaMemsetAsync(dq_acc, 0, (size_t)rows * 128 * 4, s) != cudaSuccess)
    return VSA_ERR_CUDA;
  unsigned int* status = status_word();
  if (status == nullptr) return VSA_ERR_CUDA;
  BwdArgs a{};
  a.nlse = nlse;
  a.nD = nD;
  a.bitmap = bitmap;
  a.vbs = variable_block_sizes;
  a.dq_acc = dq_acc;
  a.dk = dk;
  a.dv = dv;
  a.status = status;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.group = Hq / Hkv;
  a.Sq = Sq;
  a.Sk = Sk;
  a.nbq = nbq;
  a.nbk = nbk;
  a.scale = scale;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.wait_ns = launch_wait_ns(bwd::kWaitLimitNs);
  a.stall = g_stall.load();
  a.n_tiles = block == 64 ? (nbk + 1) / 2 : nbk;
  const long long n_ctas = (long long)B * Hkv * a.n_tiles;
  st = block == 64 ? launch_bwd<64>(dev, a, q, k, v, dout, rows, (long long)B * Hkv, n_ctas, s)
                   : launch_bwd<128>(dev, a, q, k, v, dout, rows, (long long)B * Hkv, n_ctas, s);
  if (st != VSA_OK) return st;
  if (n_ctas > 0) ++launches;
  const long long n8 = rows * 16;
  bwd_dq_kernel<<<(unsigned)((n8 + 255) / 256), 256, 0, s>>>(dq_acc, n8, scale, dq);
  if (cudaGetLastError() != cudaSuccess) return VSA_ERR_CUDA;
  t_last_launches = launches + 1;
  return VSA_OK;
}

vsa_status vsa_fwd(const vsa_bf16* q, const vsa_bf16* k, const vsa_bf16* v,
                   const int32_t* q2k_idx, const int32_t* q2k_num,
                   const int32_t* variable_block_sizes, int B, int H, int S, int D, int max_kv,
                   int block, float scale, vsa_bf16* out, float* lse, void* workspace,
                   vsa_stream_t stream) {
  const Shape p{B, H, H, S, S, D, block, scale};
  return run_lut(q, k, v, q2k_idx, q2k_num, variable_block_sizes, p, max_kv, out, lse,
                 workspace, stream, true);
}

vsa_status vsa_fwd_gqa(const vsa_bf16* q, const vsa_bf16* k, const vsa_bf16* v,
                       const int32_t* q2k_idx, const int32_t* q2k_num,
                       const int32_t* variable_block_sizes, int B, int Hq, int Hkv, int Sq,
                       int Sk, int D, int max_kv, int block, float scale, vsa_bf16* out,
                       float* lse, void* workspace, vsa_stream_t stream) {
  const Shape p{B, Hq, Hkv, Sq, Sk, D, block, scale};
  return run_lut(q, k, v, q2k_idx, q2k_num, variable_block_sizes, p, max_kv, out, lse,
                 workspace, stream, false);
}

size_t vsa_split_workspace_bytes(int B, int Hq, int Sq, int block, int num_splits) {
  if (B < 0 || Hq < 0 || Sq < 0 || (block != 64 && block != 128) || num_splits < 1 ||
      Sq % block != 0)
    return 0;
  const long long nbq = Sq / block;
  const long long items = (long long)B * Hq * (block == 64 ? (nbq + 1) / 2 : nbq);
  return kSchedBytes + (size_t)(items * num_splits) * kPartFloats * sizeof(float);
}

vsa_status vsa_fwd_split(const vsa_bf16* q, const vsa_bf16* k, const vsa_bf16* v,
                         const int32_t* q2k_idx, const int32_t* q2k_num,
                         const int32_t* variable_block_sizes, int B, int Hq, int Hkv, int Sq,
                         int Sk, int D, int max_kv, int block, float scale, int num_splits,
                         vsa_bf16* out, float* lse, void* workspace, size_t workspace_bytes,
                         vsa_stream_t stream) {
  t_last_launches = 0;
  if (num_splits < 1 || num_splits > VSA_MAX_SPLITS) return VSA_ERR_INVALID_ARG;
  const Shape p{B, Hq, Hkv, Sq, Sk, D, block, scale};
  return run_lut(q, k, v, q2k_idx, q2k_num, variable_block_sizes, p, max_kv, out, lse,
                 workspace, stream, false, num_splits, workspace_bytes);
}

vsa_status jenga_fwd(const vsa_bf16* q, const vsa_bf16* k, const vsa_bf16* v,
                     const int8_t* mask_bitmap, int B, int H, int S, int D, int block_q,
                     int block_k, float scale, vsa_bf16* out, float* lse, void* workspace,
                     vsa_stream_t stream) {
  t_last_launches = 0;
  if (block_q != block_k) return VSA_ERR_UNSUPPORTED;
  const Shape p{B, H, H, S, S, D, block_k, scale};
  return run_map(q, k, v, mask_bitmap, 0, nullptr, p, out, lse, workspace, stream);
}

vsa_status vsa_fwd_from_mask(const vsa_bf16* q, const vsa_bf16* k, const vsa_bf16* v,
                             const int8_t* block_map, int map_shared,
                             const int32_t* variable_block_sizes, int B, int Hq, int Hkv,
                             int Sq, int Sk, int D, int block, float scale, vsa_bf16* out,
                             float* lse, void* workspace, vsa_stream_t stream) {
  const Shape p{B, Hq, Hkv, Sq, Sk, D, block, scale};
  const long long stride =
      map_shared ? 0 : (block > 0 ? (long long)(Sq / block) * (Sk / block) : 0);
  return run_map(q, k, v, block_map, stride, variable_block_sizes, p, out, lse, workspace,
                 stream);
}

vsa_status vsa_lut_to_bitmap(const int32_t* q2k_idx, const int32_t* q2k_num, int rows,
                             int max_kv, int nb, int8_t* bitmap, vsa_stream_t stream) {
  if (rows < 0 || nb < 1 || max_kv < 1) return VSA_ERR_INVALID_ARG;
  if (rows == 0) return VSA_OK;
  if (!q2k_idx || !q2k_num || !bitmap) return VSA_ERR_INVALID_ARG;
  lut_to_bitmap_kernel<<<rows, 128, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      q2k_idx, q2k_num, max_kv, nb, bitmap);
  return cudaGetLastError() == cudaSuccess ? VSA_OK : VSA_ERR_CUDA;
}

vsa_status vsa_bitmap_to_lut(const int8_t* bitmap, int rows, int nb, int max_kv,
                             int32_t* q2k_idx, int32_t* q2k_num, vsa_stream_t stream) {
  if (rows < 0 || nb < 1 || max_kv < 1) return VSA_ERR_INVALID_ARG;
  if (rows == 0) return VSA_OK;
  if (!bitmap || !q2k_idx || !q2k_num) return VSA_ERR_INVALID_ARG;
  const int warps = 8;
  const int grid = (rows + warps - 1) / warps;
  bitmap_to_lut_kernel<<<grid, warps * 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      bitmap, rows, nb, max_kv, q2k_idx, q2k_num);
  return cudaGetLastError() == cudaSuccess ? VSA_OK : VSA_ERR_CUDA;
}

vsa_status vsa_fwd_from_host(const vsa_bf16* h_q, const vsa_bf16* h_k, const vsa_bf16* h_v,
                             const int32_t* h_q2k_idx, const int32_t* h_q2k_num,
                             const int32_t* h_variable_block_sizes, int B, int H, int S, int D,
                             int max_kv, int block, float scale, vsa_bf16* h_out, float* h_lse,
                             vsa_bf16* d_q, vsa_bf16* d_k, vsa_bf16* d_v, int32_t* d_q2k_idx,
                             int32_t* d_q2k_num, int32_t* d_variable_block_sizes,
                             vsa_bf16* d_out, float* d_lse, void* workspace,
                             vsa_stream_t stream) {
  t_last_launches = 0;
  if (B < 0 || H < 0 || S < 0 || D != VSA_HEAD_DIM || (block != 64 && block != 128) ||
      S % block != 0 || max_kv < 1)
    return (D != VSA_HEAD_DIM || (block != 64 && block != 128)) ? VSA_ERR_UNSUPPORTED
                                                                : VSA_ERR_INVALID_ARG;
  const size_t rows = (size_t)B * H * S;
  if (rows == 0) return VSA_OK;
  if (!h_q || !h_k || !h_v || !h_q2k_idx || !h_q2k_num || !h_variable_block_sizes || !h_out ||
      (h_lse && !d_lse))
    return VSA_ERR_INVALID_ARG;
  const size_t nb = (size_t)S / block;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // validate the device-side arguments before any copy is enqueued
  DeviceInfo* dev = nullptr;
  bool nothing = false;
  const Shape shape{B, H, H, S, S, D, block, scale};
  vsa_status st =
      check_shape(d_q, d_k, d_v, d_out, h_lse ? d_lse : nullptr, shape, &dev, &nothing);
  if (st != VSA_OK) return st;
  if (!d_q2k_idx || !d_q2k_num || !d_variable_block_sizes) return VSA_ERR_INVALID_ARG;
  if (!workspace_ok(workspace)) return VSA_ERR_INVALID_ARG;
  st = block == 64 ? prepare_fwd<64, false>(dev, 0) : prepare_fwd<128, false>(dev, 1);
  if (st != VSA_OK) return st;
  if (status_word() == nullptr) return VSA_ERR_CUDA;
  HostPipe* pipe = nullptr;
  st = host_pipe(&pipe);
  if (st != VSA_OK) return st;

  // Chunks of consecutive (b, h) heads: chunk c's inputs are copied on the input stream,
  // its forward runs on the caller's stream once they have landed, and its out / lse go
  // back on the output stream once the forward is done, so one chunk's copies overlap
  // another chunk's forward.  Both internal streams fork from `stream` and join it again.
  const int bh = B * H;
  const size_t head_bytes = (size_t)S * D * 2, lut_head = nb * (size_t)max_kv, num_head = nb;
  const size_t in_bytes = (size_t)bh * 3 * head_bytes;
  long long want = (long long)((in_bytes + kHostChunkBytes - 1) / kHostChunkBytes);
  want = want < 1 ? 1 : (want > kHostChunks ? kHostChunks : want);
  const int n_chunks = (int)(want < bh ? want : bh);
  std::lock_guard<std::mutex> lk(pipe->mu);
  // on an error after the fork, still join both internal streams back into `stream`
  auto fail = [&] {
    cudaEventRecord(pipe->ev_join, pipe->s_out);
    cudaEventRecord(pipe->ev_join_in, pipe->s_in);
    cudaStreamWaitEvent(s, pipe->ev_join, 0);
    cudaStreamWaitEvent(s, pipe->ev_join_in, 0);
    return VSA_ERR_CUDA;
  };
  if (cudaEventRecord(pipe->ev_fork, s) != cudaSuccess ||
      cudaStreamWaitEvent(pipe->s_in, pipe->ev_fork, 0) != cudaSuccess ||
      cudaStreamWaitEvent(pipe->s_out, pipe->ev_fork, 0) != cudaSuccess)
    return fail();
  if (cudaMemcpyAsync(d_variable_block_sizes, h_variable_block_sizes, nb * 4,
                      cudaMemcpyHostToDevice, pipe->s_in) != cudaSuccess)
    return fail();
  int launches = 0;
  for (int c = 0; c < n_chunks; ++c) {
    const int h0 = (int)((long long)bh * c / n_chunks), h1 = (int)((long long)bh * (c + 1) / n_chunks);
    const int nh = h1 - h0;
    const size_t t0 = (size_t)h0 * head_bytes, tb = (size_t)nh * head_bytes;
    auto in = [&](void* dst, const void* src, size_t off, size_t n) {
      return cudaMemcpyAsync(static_cast<uint8_t*>(dst) + off,
                             static_cast<const uint8_t*>(src) + off, n, cudaMemcpyHostToDevice,
                             pipe->s_in) == cudaSuccess;
    };
    if (!in(d_q, h_q, t0, tb) || !in(d_k, h_k, t0, tb) || !in(d_v, h_v, t0, tb) ||
        !in(d_q2k_idx, h_q2k_idx, (size_t)h0 * lut_head * 4, (size_t)nh * lut_head * 4) ||
        !in(d_q2k_num, h_q2k_num, (size_t)h0 * num_head * 4, (size_t)nh * num_head * 4) ||
        cudaEventRecord(pipe->ev_in[c], pipe->s_in) != cudaSuccess ||
        cudaStreamWaitEvent(s, pipe->ev_in[c], 0) != cudaSuccess)
      return fail();
    const size_t e0 = (size_t)h0 * S * D, r0 = (size_t)h0 * S;
    st = vsa_fwd(d_q + e0, d_k + e0, d_v + e0, d_q2k_idx + (size_t)h0 * lut_head,
                 d_q2k_num + (size_t)h0 * num_head, d_variable_block_sizes, 1, nh, S, D, max_kv,
                 block, scale, d_out + e0, h_lse ? d_lse + r0 : nullptr, workspace, stream);
    if (st != VSA_OK) {
      fail();
      return st;
    }
    launches += t_last_launches;
    if (cudaEventRecord(pipe->ev_done[c], s) != cudaSuccess ||
        cudaStreamWaitEvent(pipe->s_out, pipe->ev_done[c], 0) != cudaSuccess ||
        cudaMemcpyAsync(reinterpret_cast<uint8_t*>(h_out) + t0,
                        reinterpret_cast<const uint8_t*>(d_out) + t0, tb, cudaMemcpyDeviceToHost,
                        pipe->s_out) != cudaSuccess)
      return fail();
    if (h_lse && cudaMemcpyAsync(h_lse + r0, d_lse + r0, (size_t)nh * S * 4,
                                 cudaMemcpyDeviceToHost, pipe->s_out) != cudaSuccess)
      return fail();
  }
  if (cudaEventRecord(pipe->ev_join, pipe->s_out) != cudaSuccess ||
      cudaEventRecord(pipe->ev_join_in, pipe->s_in) != cudaSuccess ||
      cudaStreamWaitEvent(s, pipe->ev_join, 0) != cudaSuccess ||
      cudaStreamWaitEvent(s, pipe->ev_join_in, 0) != cudaSuccess)
    return fail();
  t_last_launches = launches;
  return VSA_OK;
}

vsa_status vsa_device_status(vsa_stream_t stream, unsigned int* detail) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return VSA_ERR_CUDA;
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof v) != cudaSuccess ||
      cudaMemcpyToSymbol(g_status, &zero, sizeof zero) != cudaSuccess)
    return VSA_ERR_CUDA;
  if (detail) *detail = v;
  return v == 0 ? VSA_OK : VSA_ERR_DEVICE_TIMEOUT;
}

int vsa_last_launch_count(void) { return t_last_launches; }

void vsa_set_wait_limit_ns(unsigned long long ns) { g_wait_ns.store(ns); }

void vsa_set_stall_test(int enable) { g_stall.store(enable ? 1 : 0); }

}  // extern "C"

// ------------------------------------------------------------------ allocation-free entry
// Scheduling scratch of vsa_fwd_noalloc: a file-scope device array used in place of the
// caller-provided workspace of vsa_fwd.  Every GPU that loads this library holds these
// VSA_NOALLOC_SCRATCH_BYTES bytes until the process exits; all calls on a device share
// them.
static __device__ __align__(256) unsigned int g_noalloc_scratch[VSA_NOALLOC_SCRATCH_BYTES / 4];

namespace {
// The array's device address, set up once per device context with that device current.
// Keyed by the context's unique id: a cudaDeviceReset (or anything else that destroys and
// recreates the context) reloads the module at a possibly different address, and the
// next call then repeats the set-up instead of using a stale pointer.
struct NoallocSlot {
  unsigned long long ctx_id = 0;
  void* addr = nullptr;
};
NoallocSlot g_noalloc[64];

bool current_context_id(unsigned long long* id) {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  if (get_current == nullptr || get_id == nullptr) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

// Every check vsa_fwd makes before it enqueues anything -- arguments, device, kernel
// attributes and register pool, the status word -- repeated here so that a call vsa_fwd
// would reject enqueues nothing, not even the scratch reset.
vsa_status noalloc_checks(const vsa_bf16* q, const vsa_bf16* k, const vsa_bf16* v,
                          const int32_t* q2k_idx, const int32_t* q2k_num,
                          const int32_t* vbs, int B, int H, int S, int D, int max_kv,
                          int block, float scale, const vsa_bf16* out, const float* lse,
                          bool* nothing) {
  DeviceInfo* dev = nullptr;
  const Shape p{B, H, H, S, S, D, block, scale};
  vsa_status st = check_shape(q, k, v, out, lse, p, &dev, nothing);
  if (st != VSA_OK || *nothing) return st;
  if (max_kv < 1) return VSA_ERR_INVALID_ARG;
  if (!q2k_idx || !q2k_num || !vbs) return VSA_ERR_INVALID_ARG;
  st = block == 64 ? prepare_fwd<64, false>(dev, 0) : prepare_fwd<128, false>(dev, 1);
  if (st != VSA_OK) return st;
  return status_word() == nullptr ? VSA_ERR_CUDA : VSA_OK;
}
}  // namespace

extern "C" {

vsa_status vsa_fwd_noalloc(const vsa_bf16* q, const vsa_bf16* k, const vsa_bf16* v,
                           const int32_t* q2k_idx, const int32_t* q2k_num,
                           const int32_t* variable_block_sizes, int B, int H, int S, int D,
                           int max_kv, int block, float scale, vsa_bf16* out, float* lse,
                           vsa_stream_t stream) {
  t_last_launches = 0;
  // the scratch this call needs must fit the static array
  if (vsa_workspace_bytes() > (size_t)VSA_NOALLOC_SCRATCH_BYTES) return VSA_ERR_UNSUPPORTED;
  bool nothing = false;
  vsa_status st = noalloc_checks(q, k, v, q2k_idx, q2k_num, variable_block_sizes, B, H, S, D,
                                 max_kv, block, scale, out, lse, &nothing);
  if (st != VSA_OK || nothing) return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return VSA_ERR_CUDA;
  void* scratch = nullptr;
  {
    // set-up, once per device (context), with that device current: the array's address
    if (cudaSetDevice(dev) != cudaSuccess) return VSA_ERR_CUDA;
    unsigned long long ctx = 0;
    if (!current_context_id(&ctx)) return VSA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    NoallocSlot& slot = g_noalloc[dev];
    if (slot.addr == nullptr || slot.ctx_id != ctx) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
        return VSA_ERR_CUDA;
      slot.addr = p;
      slot.ctx_id = ctx;
    }
    scratch = slot.addr;
  }
  // the array keeps whatever the previous call left: the scheduling counters must start
  // at zero, so clear them in stream order before the kernel
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(scratch, 0, vsa_workspace_bytes(), s) != cudaSuccess) return VSA_ERR_CUDA;
  st = vsa_fwd(q, k, v, q2k_idx, q2k_num, variable_block_sizes, B, H, S, D, max_kv, block,
               scale, out, lse, scratch, stream);
  return st;
}

const char* vsa_status_str(vsa_status s) {
  switch (s) {
    case VSA_OK: return "ok";
    case VSA_ERR_INVALID_ARG: return "invalid argument";
    case VSA_ERR_UNSUPPORTED: return "unsupported configuration";
    case VSA_ERR_CUDA: return "CUDA runtime error";
    case VSA_ERR_DEVICE_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

}  // extern "C"
