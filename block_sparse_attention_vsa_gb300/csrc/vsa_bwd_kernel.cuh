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
// Structure:
//   bwd_prep_kernel   D_i for every query row (one warp per row).
//   bwd_kv_kernel     one CTA per (batch, key/value head, key block): K and V of the block
//                     stay in SMEM; dK and dV accumulate in tensor-core fragments while the
//                     CTA walks every (query head of the group, query block) that selects
//                     the key block (a column of the 0/1 block map, compacted into an SMEM
//                     list), 64 (block 64) or 32 (block 128) query rows a step, the next
//                     step's rows copied in asynchronously while the current one computes:
//                     S = Q K^T and dP = dO V^T (tensor cores), P and dS element-wise in
//                     SMEM, then dV += P^T dO, dK += dS^T Q and dQ_part = dS K, the last
//                     added to an fp32 dQ accumulator with atomics (several key blocks feed
//                     every query row).
//   bwd_dq_kernel     fp32 dQ accumulator -> bf16 dq.
// The contractions use the warp-level bf16 tensor-core path (16x16x16 fragments, fp32
// accumulation).
#pragma once

#include <cuda_bf16.h>
#include <mma.h>

#include <cstdint>

namespace vsa {

// D_i = sum_d dout[i][d] * out[i][d] for rows rows; one warp per row, 4 elements per lane.
__global__ void __launch_bounds__(256) bwd_prep_kernel(const uint16_t* __restrict__ out,
                                                       const uint16_t* __restrict__ dout,
                                                       long long rows, float* __restrict__ Dv) {
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
  if (lane == 0) Dv[r] = acc;
}

// Four consecutive fp32 atomic adds as one vector reduction (16-byte aligned address).
__device__ __forceinline__ void red_add_v4(float* addr, float4 x) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(x.x), "f"(x.y),
               "f"(x.z), "f"(x.w)
               : "memory");
}

// fp32 dQ accumulator -> bf16 (round to nearest even), 8 elements per thread.
__global__ void __launch_bounds__(256) bwd_dq_kernel(const float* __restrict__ acc,
                                                     long long n8, uint16_t* __restrict__ dq) {
  const long long i = (long long)blockIdx.x * 256 + threadIdx.x;
  if (i >= n8) return;
  const float4 a = reinterpret_cast<const float4*>(acc)[2 * i];
  const float4 b = reinterpret_cast<const float4*>(acc)[2 * i + 1];
  uint4 o;
  o.x = pack_bf16x2(a.x, a.y);
  o.y = pack_bf16x2(a.z, a.w);
  o.z = pack_bf16x2(b.x, b.y);
  o.w = pack_bf16x2(b.z, b.w);
  reinterpret_cast<uint4*>(dq)[i] = o;
}

struct BwdArgs {
  const uint16_t *q, *k, *v, *dout;
  const float* lse;         // [B*Hq*Sq], base 2, from the forward
  const float* Dv;          // [B*Hq*Sq]
  const int8_t* bitmap;     // [B*Hq*nbq, nbk] 0/1 block map
  const int32_t* vbs;       // [nbk] or null
  float* dq_acc;            // [B*Hq*Sq, 128] fp32, zeroed
  uint16_t *dk, *dv;        // [B*Hkv*Sk, 128] bf16
  int Hq, Hkv, group, Sq, Sk, nbq, nbk;
  float scale, scale_log2;
};

template <int BLOCK>
struct BwdCfg {
  static constexpr int kWarps = 16;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kMq = BLOCK == 128 ? 32 : 64;  // query rows per step
  static constexpr int kLdH = 128 + 8;               // bf16 row pitch of K, V, Q, dO tiles
  static constexpr int kLdP = BLOCK + 8;             // bf16 row pitch of P, dS
  static constexpr int kLdS = BLOCK + 4;             // fp32 row pitch of S, dP
  static constexpr int kLdO = 128 + 4;               // fp32 row pitch of dQ / dK / dV staging
  static constexpr int kMaxSteps = 2048;             // (query head, query block) list chunk
  static constexpr size_t kQBytes = (size_t)kMq * kLdH * 2;
  static constexpr size_t kOffK = 0;
  static constexpr size_t kOffV = kOffK + (size_t)BLOCK * kLdH * 2;
  static constexpr size_t kOffQ = kOffV + (size_t)BLOCK * kLdH * 2;   // Q[2]
  static constexpr size_t kOffDO = kOffQ + 2 * kQBytes;                // dO[2]
  static constexpr size_t kOffF = kOffDO + 2 * kQBytes;               // S | dP, fp32
  static constexpr size_t kFBytesSd = (size_t)2 * kMq * kLdS * 4;
  static constexpr size_t kFBytesO = (size_t)(BLOCK > kMq ? BLOCK : kMq) * kLdO * 4;
  static constexpr size_t kFBytes = kFBytesSd > kFBytesO ? kFBytesSd : kFBytesO;
  static constexpr size_t kOffP = kOffF + kFBytes;
  static constexpr size_t kOffDS = kOffP + (size_t)kMq * kLdP * 2;
  static constexpr size_t kOffRow = kOffDS + (size_t)kMq * kLdP * 2;  // [2] x (lse, D)[kMq]
  static constexpr size_t kOffList = kOffRow + 2 * 2 * kMq * 4;
  static constexpr size_t kSmem = kOffList + (size_t)kMaxSteps * 4 + 16;
  static constexpr int kTilesKV = (BLOCK / 16) * 8;                  // dK or dV 16x16 tiles
  static constexpr int kAccPerWarp = kTilesKV / kWarps;              // 2 or 4
  static constexpr int kTilesQ = (kMq / 16) * 8;                     // dQ part tiles
  static constexpr int kQPerWarp = kTilesQ / kWarps;                 // 2 or 1
  static constexpr int kSCols = BLOCK / 16;                          // S / dP column tiles
};
static_assert(BwdCfg<64>::kQPerWarp >= 1 && BwdCfg<128>::kQPerWarp >= 1, "dQ tiles per warp");
static_assert(BwdCfg<64>::kSmem <= 227 * 1024 && BwdCfg<128>::kSmem <= 227 * 1024,
              "backward SMEM");

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// rows x 128 bf16 from global (row stride 128) into SMEM with row pitch kLdH, 16 B a time
template <int BLOCK>
__device__ __forceinline__ void load_rows(uint16_t* dst, const uint16_t* src, int rows) {
  using C = BwdCfg<BLOCK>;
  for (int i = threadIdx.x; i < rows * 16; i += C::kThreads) {
    const int r = i >> 4, c = i & 15;
    reinterpret_cast<uint4*>(dst + r * C::kLdH)[c] = reinterpret_cast<const uint4*>(src + r * 128)[c];
  }
}

// Asynchronous copy of one step's inputs: kMq rows of Q and dO, their lse and D.
template <int BLOCK>
__device__ __forceinline__ void prefetch_step(uint8_t* smem, int buf, const BwdArgs& a,
                                              long long qrow0) {
  using C = BwdCfg<BLOCK>;
  uint8_t* qd = smem + C::kOffQ + buf * C::kQBytes;
  uint8_t* od = smem + C::kOffDO + buf * C::kQBytes;
  for (int i = threadIdx.x; i < C::kMq * 16; i += C::kThreads) {
    const int r = i >> 4, c = i & 15;
    cp_async16(qd + (r * C::kLdH + c * 8) * 2, a.q + (qrow0 + r) * 128 + c * 8);
    cp_async16(od + (r * C::kLdH + c * 8) * 2, a.dout + (qrow0 + r) * 128 + c * 8);
  }
  float* row = reinterpret_cast<float*>(smem + C::kOffRow) + buf * 2 * C::kMq;
  for (int i = threadIdx.x; i < C::kMq / 4; i += C::kThreads) {
    cp_async16(row + 4 * i, a.lse + qrow0 + 4 * i);
    cp_async16(row + C::kMq + 4 * i, a.Dv + qrow0 + 4 * i);
  }
  cp_async_commit();
}

template <int BLOCK>
__global__ void __launch_bounds__(BwdCfg<BLOCK>::kThreads, 1) bwd_kv_kernel(const BwdArgs a) {
  using namespace nvcuda;
  using C = BwdCfg<BLOCK>;
  using FragA = wmma::fragment<wmma::matrix_a, 16, 16, 16, __nv_bfloat16, wmma::row_major>;
  using FragAc = wmma::fragment<wmma::matrix_a, 16, 16, 16, __nv_bfloat16, wmma::col_major>;
  using FragB = wmma::fragment<wmma::matrix_b, 16, 16, 16, __nv_bfloat16, wmma::row_major>;
  using FragBc = wmma::fragment<wmma::matrix_b, 16, 16, 16, __nv_bfloat16, wmma::col_major>;
  using FragC = wmma::fragment<wmma::accumulator, 16, 16, 16, float>;
  extern __shared__ __align__(128) uint8_t smem_b[];
  __nv_bfloat16* Ks = reinterpret_cast<__nv_bfloat16*>(smem_b + C::kOffK);
  __nv_bfloat16* Vs = reinterpret_cast<__nv_bfloat16*>(smem_b + C::kOffV);
  float* Sf = reinterpret_cast<float*>(smem_b + C::kOffF);
  float* dPf = Sf + C::kMq * C::kLdS;
  float* Of = Sf;  // dQ part / dK / dV staging (after S and dP are consumed)
  __nv_bfloat16* Pb = reinterpret_cast<__nv_bfloat16*>(smem_b + C::kOffP);
  __nv_bfloat16* dSb = reinterpret_cast<__nv_bfloat16*>(smem_b + C::kOffDS);
  uint32_t* steps = reinterpret_cast<uint32_t*>(smem_b + C::kOffList);
  int* n_steps = reinterpret_cast<int*>(smem_b + C::kOffList + (size_t)C::kMaxSteps * 4);
  const int warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31;

  const int kb = blockIdx.x % a.nbk;
  const int bkv = blockIdx.x / a.nbk;  // b * Hkv + hk
  const int b = bkv / a.Hkv, hk = bkv - b * a.Hkv;
  const long long krow0 = (long long)bkv * a.Sk + (long long)kb * BLOCK;
  int vk = BLOCK;
  if (a.vbs != nullptr) {
    vk = a.vbs[kb];
    vk = vk < 0 ? 0 : (vk > BLOCK ? BLOCK : vk);
  }
  load_rows<BLOCK>(reinterpret_cast<uint16_t*>(Ks), a.k + krow0 * 128, BLOCK);
  load_rows<BLOCK>(reinterpret_cast<uint16_t*>(Vs), a.v + krow0 * 128, BLOCK);

  // this warp's dK and dV tiles: key-row tiles (warp / 8) * kAccPerWarp + i, d column
  // tile warp % 8
  FragC dK[C::kAccPerWarp], dV[C::kAccPerWarp];
#pragma unroll
  for (int i = 0; i < C::kAccPerWarp; ++i) {
    wmma::fill_fragment(dK[i], 0.0f);
    wmma::fill_fragment(dV[i], 0.0f);
  }

  constexpr int kSub = BLOCK / C::kMq;  // steps per query block
  int scan_h = 0, scan_qb = 0;          // warp 0's position in the (head, query block) scan
  while (true) {
    // ---- the next chunk of (query head, query block) pairs selecting this key block:
    // a column of the block map, compacted in order by warp 0
    __syncthreads();  // the previous chunk is done with the list
    if (warp == 0) {
      int cnt = 0;
      while (scan_h < a.group && cnt + 32 <= C::kMaxSteps) {
        const long long bh = (long long)b * a.Hq + hk * a.group + scan_h;
        const int qb = scan_qb + (int)lane;
        const bool sel = qb < a.nbq && a.bitmap[(bh * a.nbq + qb) * (long long)a.nbk + kb] != 0;
        const uint32_t ballot = __ballot_sync(0xffffffffu, sel);
        if (sel) steps[cnt + __popc(ballot & ((1u << lane) - 1u))] = ((uint32_t)scan_h << 20) | qb;
        cnt += __popc(ballot);
        scan_qb += 32;
        if (scan_qb >= a.nbq) {
          scan_qb = 0;
          ++scan_h;
        }
      }
      if (lane == 0) *n_steps = cnt;
    }
    __syncthreads();
    const int n = *n_steps;
    if (n == 0) break;
    const int total = n * kSub;
    auto step_row = [&](int s) -> long long {
      const uint32_t e = steps[s / kSub];
      const long long bh = (long long)b * a.Hq + hk * a.group + (int)(e >> 20);
      return bh * a.Sq + (long long)(e & 0xFFFFFu) * BLOCK + (s % kSub) * C::kMq;
    };
    prefetch_step<BLOCK>(smem_b, 0, a, step_row(0));
    for (int s = 0; s < total; ++s) {
      const int buf = s & 1;
      const long long qrow0 = step_row(s);
      if (s + 1 < total) {
        prefetch_step<BLOCK>(smem_b, buf ^ 1, a, step_row(s + 1));
        cp_async_wait<1>();
      } else {
        cp_async_wait<0>();
      }
      __syncthreads();  // this step's inputs have landed for every thread
      const __nv_bfloat16* Qs =
          reinterpret_cast<const __nv_bfloat16*>(smem_b + C::kOffQ + buf * C::kQBytes);
      const __nv_bfloat16* dOs =
          reinterpret_cast<const __nv_bfloat16*>(smem_b + C::kOffDO + buf * C::kQBytes);
      const float* lse_s = reinterpret_cast<const float*>(smem_b + C::kOffRow) + buf * 2 * C::kMq;
      const float* D_s = lse_s + C::kMq;
      // S = Q K^T and dP = dO V^T: (kMq / 16) x (BLOCK / 16) tiles of each; a warp takes
      // two column tiles of one row tile of one of them, reusing its A fragment
      {
        static_assert(2 * (C::kMq / 16) * C::kSCols == 2 * C::kWarps, "S tiles per warp");
        const int half = C::kWarps / 2;
        const bool isdp = warp >= half;
        const int idx = warp - (isdp ? half : 0);
        const int tr = idx / (C::kSCols / 2), tc0 = 2 * (idx % (C::kSCols / 2));
        const __nv_bfloat16* A = isdp ? dOs : Qs;
        const __nv_bfloat16* Bm = isdp ? Vs : Ks;
        FragC acc0, acc1;
        wmma::fill_fragment(acc0, 0.0f);
        wmma::fill_fragment(acc1, 0.0f);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          FragA fa;
          FragBc fb0, fb1;  // K^T: column-major views of the row-major K tile
          wmma::load_matrix_sync(fa, A + tr * 16 * C::kLdH + kk * 16, C::kLdH);
          wmma::load_matrix_sync(fb0, Bm + tc0 * 16 * C::kLdH + kk * 16, C::kLdH);
          wmma::load_matrix_sync(fb1, Bm + (tc0 + 1) * 16 * C::kLdH + kk * 16, C::kLdH);
          wmma::mma_sync(acc0, fa, fb0, acc0);
          wmma::mma_sync(acc1, fa, fb1, acc1);
        }
        float* dst = (isdp ? dPf : Sf) + tr * 16 * C::kLdS + tc0 * 16;
        wmma::store_matrix_sync(dst, acc0, C::kLdS, wmma::mem_row_major);
        wmma::store_matrix_sync(dst + 16, acc1, C::kLdS, wmma::mem_row_major);
      }
      __syncthreads();
      // P and dS (dS carries the softmax scale of dq and dk)
      for (int i = threadIdx.x; i < C::kMq * BLOCK; i += C::kThreads) {
        const int r = i / BLOCK, j = i - r * BLOCK;
        const float l2 = lse_s[r];
        const bool valid = j < vk && l2 > -3.0e38f;  // tail keys; rows with no key
        const float p = valid ? exp2f(fmaf(Sf[r * C::kLdS + j], a.scale_log2, -l2)) : 0.0f;
        const float ds = p * (dPf[r * C::kLdS + j] - D_s[r]) * a.scale;
        Pb[r * C::kLdP + j] = __float2bfloat16_rn(p);
        dSb[r * C::kLdP + j] = __float2bfloat16_rn(ds);
      }
      __syncthreads();
      // dV += P^T dO and dK += dS^T Q, k over the kMq query rows: this warp's tiles share
      // one d column tile (so one dO and one Q fragment per k step)
      {
        const int tc = warp % 8, tr0 = (warp / 8) * C::kAccPerWarp;
#pragma unroll
        for (int kk = 0; kk < C::kMq / 16; ++kk) {
          FragB fo, fq;
          wmma::load_matrix_sync(fo, dOs + kk * 16 * C::kLdH + tc * 16, C::kLdH);
          wmma::load_matrix_sync(fq, Qs + kk * 16 * C::kLdH + tc * 16, C::kLdH);
#pragma unroll
          for (int i = 0; i < C::kAccPerWarp; ++i) {
            FragAc fp, fds;  // P^T, dS^T: column-major views of row-major P, dS
            wmma::load_matrix_sync(fp, Pb + kk * 16 * C::kLdP + (tr0 + i) * 16, C::kLdP);
            wmma::mma_sync(dV[i], fp, fo, dV[i]);
            wmma::load_matrix_sync(fds, dSb + kk * 16 * C::kLdP + (tr0 + i) * 16, C::kLdP);
            wmma::mma_sync(dK[i], fds, fq, dK[i]);
          }
        }
      }
      // dQ part = dS K, k over the BLOCK keys (S / dP are dead): this warp's tiles share one
      // row tile (one dS fragment per k step)
      {
        const int base = warp * C::kQPerWarp, tr = base / 8, tc0 = base % 8;
        FragC acc[C::kQPerWarp];
#pragma unroll
        for (int j = 0; j < C::kQPerWarp; ++j) wmma::fill_fragment(acc[j], 0.0f);
#pragma unroll
        for (int kk = 0; kk < BLOCK / 16; ++kk) {
          FragA fa;
          wmma::load_matrix_sync(fa, dSb + tr * 16 * C::kLdP + kk * 16, C::kLdP);
#pragma unroll
          for (int j = 0; j < C::kQPerWarp; ++j) {
            FragB fb;
            wmma::load_matrix_sync(fb, Ks + kk * 16 * C::kLdH + (tc0 + j) * 16, C::kLdH);
            wmma::mma_sync(acc[j], fa, fb, acc[j]);
          }
        }
#pragma unroll
        for (int j = 0; j < C::kQPerWarp; ++j)
          wmma::store_matrix_sync(Of + tr * 16 * C::kLdO + (tc0 + j) * 16, acc[j], C::kLdO,
                                  wmma::mem_row_major);
      }
      __syncthreads();
      float* dst = a.dq_acc + qrow0 * 128;
      for (int i = threadIdx.x; i < C::kMq * 32; i += C::kThreads) {  // 4 floats a time
        const int r = i >> 5, c4 = (i & 31) * 4;
        const float4 x = *reinterpret_cast<const float4*>(Of + r * C::kLdO + c4);
        red_add_v4(dst + r * 128 + c4, x);
      }
      __syncthreads();  // Of, P, dS and this step's buffer are free again
    }
  }
  // dK, dV -> bf16, through the fp32 staging area
  for (int which = 0; which < 2; ++which) {
#pragma unroll
    for (int i = 0; i < C::kAccPerWarp; ++i) {
      const int tr = (warp / 8) * C::kAccPerWarp + i, tc = warp % 8;
      wmma::store_matrix_sync(Of + tr * 16 * C::kLdO + tc * 16, which ? dV[i] : dK[i], C::kLdO,
                              wmma::mem_row_major);
    }
    __syncthreads();
    uint16_t* dst = (which ? a.dv : a.dk) + krow0 * 128;
    for (int i = threadIdx.x; i < BLOCK * 64; i += C::kThreads) {
      const int r = i >> 6, c2 = (i & 63) * 2;
      reinterpret_cast<uint32_t*>(dst + r * 128)[c2 >> 1] =
          pack_bf16x2(Of[r * C::kLdO + c2], Of[r * C::kLdO + c2 + 1]);
    }
    __syncthreads();
  }
}

}  // namespace vsa
