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
//                     list), 32 query rows a step, the next step's rows copied in
//                     asynchronously while the current one computes.  Each warp owns 16
//                     keys: S^T = K Q^T and dP^T = V dO^T land in its registers, P^T and
//                     dS^T are formed there and reused as the A operands of dV += P^T dO
//                     and dK += dS^T Q (dK, dV stay in registers); dS^T goes through SMEM
//                     for dQ_part = dS K, added to an fp32 dQ accumulator with vector
//                     reductions (several key blocks feed every query row).
//   bwd_dq_kernel     fp32 dQ accumulator -> bf16 dq.
// The contractions use the warp-level bf16 tensor-core path (mma.sync m16n8k16, fp32
// accumulation, operands through ldmatrix).
#pragma once

#include <cuda_bf16.h>

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
  static constexpr int kWarps = BLOCK / 16;          // one warp per 16 keys: 4 or 8
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kMq = 32;                     // query rows per step
  static constexpr int kLdH = 128 + 8;               // bf16 row pitch of K, V, Q, dO tiles
  static constexpr int kLdT = kMq + 8;               // bf16 row pitch of the dS^T tile
  static constexpr int kMaxSteps = 2048;             // (query head, query block) list chunk
  static constexpr size_t kQBytes = (size_t)kMq * kLdH * 2;
  static constexpr size_t kOffK = 0;
  static constexpr size_t kOffV = kOffK + (size_t)BLOCK * kLdH * 2;
  static constexpr size_t kOffQ = kOffV + (size_t)BLOCK * kLdH * 2;   // Q[2]
  static constexpr size_t kOffDO = kOffQ + 2 * kQBytes;                // dO[2]
  static constexpr size_t kOffDS = kOffDO + 2 * kQBytes;               // dS^T [BLOCK][kLdT]
  static constexpr size_t kOffRow = kOffDS + (size_t)BLOCK * kLdT * 2; // [2] x (lse, D)[kMq]
  static constexpr size_t kOffList = kOffRow + 2 * 2 * kMq * 4;
  static constexpr size_t kSmem = kOffList + (size_t)kMaxSteps * 4 + 16;
};
static_assert(BwdCfg<64>::kSmem <= 113 * 1024, "two block-64 backward CTAs per SM");
static_assert(BwdCfg<128>::kSmem <= 227 * 1024, "backward SMEM");

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

// Warp-level tensor-core primitives (the m16n8k16 bf16 mma.sync path, fp32 accumulate).
// Fragment layout with g = lane / 4, t = lane % 4: an accumulator holds rows g and g + 8,
// columns 2t and 2t + 1 of a 16 x 8 tile; an A fragment holds rows g, g + 8 and k
// columns 2t, 2t + 1, 2t + 8, 2t + 9 of a 16 x 16 tile; a B fragment k rows 2t, 2t + 1,
// 2t + 8, 2t + 9 of column g of a 16 x 8 tile.
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_addr(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_addr(p)));
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
      " {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void red_add_v2(float* addr, float x, float y) {
  asm volatile("red.global.add.v2.f32 [%0], {%1, %2};" ::"l"(addr), "f"(x), "f"(y) : "memory");
}
// ldmatrix row addresses: A (or B stored as [n][k]) from a row-major tile at (r0, c0)
__device__ __forceinline__ const __nv_bfloat16* frag_a_addr(const __nv_bfloat16* base, int ld,
                                                            int r0, int c0, uint32_t lane) {
  return base + (r0 + (int)(lane & 15)) * ld + c0 + (int)(lane >> 4) * 8;
}
// two 8-wide n tiles of B stored as [n][k]: rows n0.., k columns k0..k0+15
__device__ __forceinline__ const __nv_bfloat16* frag_bn_addr(const __nv_bfloat16* base, int ld,
                                                             int n0, int k0, uint32_t lane) {
  return base + (n0 + (int)(lane & 7) + (int)(lane >> 4) * 8) * ld + k0 + (int)((lane >> 3) & 1) * 8;
}
// two 8-wide n tiles of B stored as [k][n] (transposed load): rows k0.., columns n0..n0+15
__device__ __forceinline__ const __nv_bfloat16* frag_bk_addr(const __nv_bfloat16* base, int ld,
                                                             int k0, int n0, uint32_t lane) {
  return base + (k0 + (int)(lane & 15)) * ld + n0 + (int)(lane >> 4) * 8;
}
// A stored transposed as [k][m] (transposed load): rows k0.., columns m0..m0+15
__device__ __forceinline__ const __nv_bfloat16* frag_at_addr(const __nv_bfloat16* base, int ld,
                                                             int k0, int m0, uint32_t lane) {
  return base + (k0 + (int)(lane & 7) + (int)(lane >> 4) * 8) * ld + m0 + (int)((lane >> 3) & 1) * 8;
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
__global__ void __launch_bounds__(BwdCfg<BLOCK>::kThreads) bwd_kv_kernel(const BwdArgs a) {
  using C = BwdCfg<BLOCK>;
  extern __shared__ __align__(128) uint8_t smem_b[];
  const __nv_bfloat16* Ks = reinterpret_cast<const __nv_bfloat16*>(smem_b + C::kOffK);
  const __nv_bfloat16* Vs = reinterpret_cast<const __nv_bfloat16*>(smem_b + C::kOffV);
  __nv_bfloat16* dST = reinterpret_cast<__nv_bfloat16*>(smem_b + C::kOffDS);
  uint32_t* steps = reinterpret_cast<uint32_t*>(smem_b + C::kOffList);
  int* n_steps = reinterpret_cast<int*>(smem_b + C::kOffList + (size_t)C::kMaxSteps * 4);
  const int warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31;
  const int g = (int)(lane >> 2), tq = (int)(lane & 3);

  const int kb = blockIdx.x % a.nbk;
  const int bkv = blockIdx.x / a.nbk;  // b * Hkv + hk
  const int b = bkv / a.Hkv, hk = bkv - b * a.Hkv;
  const long long krow0 = (long long)bkv * a.Sk + (long long)kb * BLOCK;
  int vk = BLOCK;
  if (a.vbs != nullptr) {
    vk = a.vbs[kb];
    vk = vk < 0 ? 0 : (vk > BLOCK ? BLOCK : vk);
  }
  load_rows<BLOCK>(reinterpret_cast<uint16_t*>(smem_b + C::kOffK), a.k + krow0 * 128, BLOCK);
  load_rows<BLOCK>(reinterpret_cast<uint16_t*>(smem_b + C::kOffV), a.v + krow0 * 128, BLOCK);

  // this warp's 16 keys: rows 16 warp + g and + 8 of the key block
  const int key0 = 16 * warp + g, key1 = key0 + 8;
  const bool kv0 = key0 < vk, kv1 = key1 < vk;
  float dK[16][4], dV[16][4];  // [d tile of 8][fragment]
#pragma unroll
  for (int i = 0; i < 16; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) dK[i][j] = dV[i][j] = 0.0f;

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
      // ---- S^T = K Q^T and dP^T = V dO^T for this warp's 16 keys x kMq queries
      float sT[4][4], dpT[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) sT[i][j] = dpT[i][j] = 0.0f;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {  // d in steps of 16
        uint32_t ak[4], av[4];
        ldsm_x4(ak, frag_a_addr(Ks, C::kLdH, 16 * warp, 16 * kk, lane));
        ldsm_x4(av, frag_a_addr(Vs, C::kLdH, 16 * warp, 16 * kk, lane));
#pragma unroll
        for (int p = 0; p < 2; ++p) {  // query tiles 2p, 2p + 1
          uint32_t bq[4], bo[4];
          ldsm_x4(bq, frag_bn_addr(Qs, C::kLdH, 16 * p, 16 * kk, lane));
          ldsm_x4(bo, frag_bn_addr(dOs, C::kLdH, 16 * p, 16 * kk, lane));
          mma16816(sT[2 * p], ak, bq[0], bq[1]);
          mma16816(sT[2 * p + 1], ak, bq[2], bq[3]);
          mma16816(dpT[2 * p], av, bo[0], bo[1]);
          mma16816(dpT[2 * p + 1], av, bo[2], bo[3]);
        }
      }
      // ---- P^T and dS^T (dS carries the softmax scale of dq and dk), as A fragments
      uint32_t pA[2][4], dsA[2][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        float p[4], ds[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int qc = 8 * nt + 2 * tq + (j & 1);
          const float l2 = lse_s[qc];
          const bool valid = (j < 2 ? kv0 : kv1) && l2 > -3.0e38f;
          p[j] = valid ? exp2f(fmaf(sT[nt][j], a.scale_log2, -l2)) : 0.0f;
          ds[j] = p[j] * (dpT[nt][j] - D_s[qc]) * a.scale;
        }
        // accumulator (16 x 8 tile nt) -> half of the A fragment of k step nt / 2
        pA[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16x2(p[0], p[1]);
        pA[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16x2(p[2], p[3]);
        dsA[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16x2(ds[0], ds[1]);
        dsA[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16x2(ds[2], ds[3]);
        // dS^T to SMEM for dq: rows key0 / key1, query columns 8 nt + 2 tq, + 1
        *reinterpret_cast<uint32_t*>(dST + key0 * C::kLdT + 8 * nt + 2 * tq) =
            dsA[nt >> 1][(nt & 1) * 2 + 0];
        *reinterpret_cast<uint32_t*>(dST + key1 * C::kLdT + 8 * nt + 2 * tq) =
            dsA[nt >> 1][(nt & 1) * 2 + 1];
      }
      // ---- dV += P^T dO and dK += dS^T Q: k over the kMq queries, n over d
#pragma unroll
      for (int j = 0; j < C::kMq / 16; ++j) {
#pragma unroll
        for (int dp = 0; dp < 8; ++dp) {  // d tiles 2dp, 2dp + 1
          uint32_t bo[4], bq[4];
          ldsm_x4_t(bo, frag_bk_addr(dOs, C::kLdH, 16 * j, 16 * dp, lane));
          ldsm_x4_t(bq, frag_bk_addr(Qs, C::kLdH, 16 * j, 16 * dp, lane));
          mma16816(dV[2 * dp], pA[j], bo[0], bo[1]);
          mma16816(dV[2 * dp + 1], pA[j], bo[2], bo[3]);
          mma16816(dK[2 * dp], dsA[j], bq[0], bq[1]);
          mma16816(dK[2 * dp + 1], dsA[j], bq[2], bq[3]);
        }
      }
      __syncthreads();  // dS^T complete
      // ---- dQ part = dS K: query row tile rt, a range of d tiles, k over the BLOCK keys
      {
        constexpr int kRowTiles = C::kMq / 16;                 // 2
        constexpr int kDTiles = 16 / (C::kWarps / kRowTiles);  // 8 (block 64) or 4 (block 128)
        const int rt = warp % kRowTiles, d0 = (warp / kRowTiles) * kDTiles;
        float acc[kDTiles][4];
#pragma unroll
        for (int i = 0; i < kDTiles; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
#pragma unroll
        for (int kk = 0; kk < BLOCK / 16; ++kk) {
          uint32_t ad[4];
          ldsm_x4_t(ad, frag_at_addr(dST, C::kLdT, 16 * kk, 16 * rt, lane));
#pragma unroll
          for (int dp = 0; dp < kDTiles / 2; ++dp) {
            uint32_t bk[4];
            ldsm_x4_t(bk, frag_bk_addr(Ks, C::kLdH, 16 * kk, 8 * d0 + 16 * dp, lane));
            mma16816(acc[2 * dp], ad, bk[0], bk[1]);
            mma16816(acc[2 * dp + 1], ad, bk[2], bk[3]);
          }
        }
        float* dst = a.dq_acc + (qrow0 + 16 * rt + g) * 128 + 8 * d0 + 2 * tq;
#pragma unroll
        for (int i = 0; i < kDTiles; ++i) {
          red_add_v2(dst + 8 * i, acc[i][0], acc[i][1]);
          red_add_v2(dst + 8 * 128 + 8 * i, acc[i][2], acc[i][3]);
        }
      }
      __syncthreads();  // dS^T and this step's buffer are free again
    }
  }
  // dK, dV -> bf16: rows key0 / key1, d columns 8 i + 2 tq, + 1
  uint16_t* dk = a.dk + (krow0 + key0) * 128 + 2 * tq;
  uint16_t* dv = a.dv + (krow0 + key0) * 128 + 2 * tq;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    *reinterpret_cast<uint32_t*>(dk + 8 * i) = pack_bf16x2(dK[i][0], dK[i][1]);
    *reinterpret_cast<uint32_t*>(dk + 8 * 128 + 8 * i) = pack_bf16x2(dK[i][2], dK[i][3]);
    *reinterpret_cast<uint32_t*>(dv + 8 * i) = pack_bf16x2(dV[i][0], dV[i][1]);
    *reinterpret_cast<uint32_t*>(dv + 8 * 128 + 8 * i) = pack_bf16x2(dV[i][2], dV[i][3]);
  }
}

}  // namespace vsa
