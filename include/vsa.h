/*
 * vsa.h -- C ABI of the GB300 (sm_103a) block-sparse attention forward library
 * (libvsa_gb300.so).
 *
 * The operation (both entry points compute the same thing; they differ in how the
 * block selection is encoded):
 *
 *   For batch b, head h and query row i, let qb = i / block be its query block.
 *   Key j (key block kb = j / block) is attended iff kb is selected for (b, h, qb)
 *   and (j mod block) < variable_block_sizes[kb].  Over the attended keys A_i:
 *
 *     out[b,h,i,:] = sum_{j in A_i} softmax_j(scale * q_i . k_j) * v[b,h,j,:]
 *     lse[b,h,i]   = log2( sum_{j in A_i} exp(scale * q_i . k_j) )
 *                  = max_j(q_i.k_j * scale * log2 e) + log2(l)      (base 2)
 *
 *   A row with no attended key gets out = +0.0 in every element and
 *   lse = VSA_LSE_EMPTY.
 *
 *   Sources: "FastVideo block_sparse_attn_sm100a.py" -- module docstring (forward
 *   returns (out, lse), lse = max(qk*qk_scale) + log2(l), [B,H,S] fp32; 64- and
 *   128-token blocks) and is_supported docstring (BHSD bf16, head_dim 128, even
 *   number of blocks, per-row counts in [0, max_kv], padding past a row's count never
 *   read, count 0 -> zero output and a finite LSE sentinel, keys at or past a block's
 *   valid count masked); "TheRock rocke sparse_attention.py" -- module docstring (the
 *   Jenga i8 MaskBitmap[q_block, k_block], 1 = attend; the VSA per-q-block LUT of
 *   BlockCount entries) and _lds_bitmap_predicate (a nonzero byte means attend).
 *
 * Conventions shared by every entry point:
 *   - Tensors are dense and contiguous.  q, k, v, out are bf16 bit patterns laid out
 *     [B, H, S, D] (BHSD), D = VSA_HEAD_DIM = 128, 16-byte aligned.  The library
 *     never takes ownership of and never retains a pointer; it allocates nothing.
 *   - Device pointers unless the name says host.  All work is enqueued on `stream`
 *     (a cudaStream_t; NULL = the legacy default stream) and is asynchronous: the
 *     call returns once the work is enqueued.  No host-device synchronisation, no
 *     reads of tensor contents on the host.
 *   - Argument checks happen on the host before anything is enqueued; a failed check
 *     returns an error and enqueues nothing.
 *   - Metadata is int32.  LUT entries below a row's count must lie in [0, nb);
 *     entries outside that range are skipped, counts are clamped to [0, max_kv], and
 *     a block named twice in one row is attended once (set semantics).
 *   - Each kernel bounds every internal wait (about one second).  A wait that runs
 *     out records a code in a device status word and the kernel returns early; read
 *     it with vsa_device_status().
 */
#ifndef VSA_GB300_H
#define VSA_GB300_H

#include <float.h>
#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum vsa_status {
  VSA_OK = 0,
  VSA_ERR_INVALID_ARG = 1,    /* null pointer, bad shape, misaligned tensor, bad scale */
  VSA_ERR_UNSUPPORTED = 2,    /* valid but not built for: D != 128, block not 64/128,
                                 too many key blocks, device not sm_103 */
  VSA_ERR_CUDA = 3,           /* a CUDA runtime call failed (launch, copy, attribute) */
  VSA_ERR_DEVICE_TIMEOUT = 4  /* a kernel gave up on an internal wait (vsa_device_status) */
} vsa_status;

/* Finite stand-in for log2(0) written to lse for rows with no attended key:
 * -FLT_MAX, the most negative finite binary32. */
#define VSA_LSE_EMPTY (-FLT_MAX)
#define VSA_HEAD_DIM 128
/* Largest number of key blocks per sequence (Sk / block) the kernels accept. */
#define VSA_MAX_BLOCKS 2048
/* Largest num_splits vsa_fwd_split accepts. */
#define VSA_MAX_SPLITS 64

/* every entry point is exported from the shared library */
#if defined(__GNUC__)
#define VSA_API __attribute__((visibility("default")))
#else
#define VSA_API
#endif

typedef uint16_t vsa_bf16;            /* bf16 bit pattern */
typedef struct CUstream_st *vsa_stream_t; /* == cudaStream_t */

/* VSA forward.
 *   q, k, v      [B, H, S, D] bf16.
 *   q2k_idx      [B, H, nb, max_kv] int32, nb = S / block: the key blocks each query
 *                block attends; row (b, h, qb) holds its q2k_num[b, h, qb] valid entries
 *                first, anything after them (e.g. -1 padding) is never read.
 *   q2k_num      [B, H, nb] int32 valid-entry counts (0 allowed).
 *   variable_block_sizes  [nb] int32, each in [0, block]: valid keys of each key block;
 *                keys at positions >= it are masked (values are clamped to [0, block]).
 *   block        64 or 128 tokens per block; S must be a multiple.  (The FastVideo
 *                contract asks for an even nb; an odd nb is accepted as well: with block
 *                64 the last query block of each head is then computed on its own.)
 *   scale        natural-exp softmax scale (finite, > 0), typically 1/sqrt(D).
 *   out          [B, H, S, D] bf16 output; must not overlap any input.
 *   lse          [B, H, S] fp32 output (base 2), or NULL to skip it (need_lse = false).
 *   workspace    NULL, or device memory of at least vsa_workspace_bytes() bytes that
 *                is all zero before the first call; each call leaves it zero again.
 *                With a workspace, work items are handed out dynamically (better
 *                balance for uneven counts); calls sharing one workspace must not
 *                overlap on the GPU.  NULL selects a static round-robin schedule.
 * Source: "FastVideo block_sparse_attn_sm100a.py", block_sparse_attn_sm100a and
 * is_supported; "TheRock rocke sparse_attention.py", build_vsa_sparse_attention. */
VSA_API vsa_status vsa_fwd(const vsa_bf16 *q, const vsa_bf16 *k, const vsa_bf16 *v,
                   const int32_t *q2k_idx, const int32_t *q2k_num,
                   const int32_t *variable_block_sizes, int B, int H, int S, int D,
                   int max_kv, int block, float scale, vsa_bf16 *out, float *lse,
                   void *workspace, vsa_stream_t stream);

/* Jenga forward: the selection is one i8 bitmap mask_bitmap[S/block_q, S/block_k],
 * shared by every batch and head; a nonzero byte means attend.  Every key of a selected
 * block is valid (no tail mask).  block_q == block_k, 64 or 128; S a multiple of it.
 * Other arguments as vsa_fwd.
 * Source: "TheRock rocke sparse_attention.py", module docstring (Jenga bullet),
 * _stage_jenga_mask_to_lds, _lds_bitmap_predicate, build_jenga_sparse_attention. */
VSA_API vsa_status jenga_fwd(const vsa_bf16 *q, const vsa_bf16 *k, const vsa_bf16 *v,
                     const int8_t *mask_bitmap, int B, int H, int S, int D, int block_q,
                     int block_k, float scale, vsa_bf16 *out, float *lse, void *workspace,
                     vsa_stream_t stream);

/* Grouped-query and cross-length VSA forward: vsa_fwd with separate query / key-value
 * head counts and sequence lengths.
 *   q, out       [B, Hq, Sq, D] bf16;  k, v  [B, Hkv, Sk, D] bf16;  Hq a multiple of Hkv.
 *                Query head hq reads key/value head hq / (Hq / Hkv).
 *   q2k_idx      [B, Hq, Sq/block, max_kv] int32, entries in [0, Sk/block).
 *   q2k_num      [B, Hq, Sq/block] int32.
 *   variable_block_sizes  [Sk/block] int32, or NULL for full key blocks.
 *   lse          [B, Hq, Sq] fp32 or NULL.
 *   Sq and Sk are multiples of block; Sk / block <= VSA_MAX_BLOCKS.  Sk = 0 is allowed:
 *   every row is then empty (out 0, lse VSA_LSE_EMPTY).  Hq % Hkv != 0 is
 *   VSA_ERR_INVALID_ARG.  Other arguments and errors as vsa_fwd; with Hq = Hkv = H and
 *   Sq = Sk = S this is vsa_fwd.
 * Source: "TheRock rocke sparse_attention.py", JengaSparseSpec / VsaSparseSpec (separate
 * seqlen_q, seqlen_k and query / key-value head counts; the key-value head of a query
 * head, kv_head_idx). */
VSA_API vsa_status vsa_fwd_gqa(const vsa_bf16 *q, const vsa_bf16 *k, const vsa_bf16 *v,
                               const int32_t *q2k_idx, const int32_t *q2k_num,
                               const int32_t *variable_block_sizes, int B, int Hq, int Hkv,
                               int Sq, int Sk, int D, int max_kv, int block, float scale,
                               vsa_bf16 *out, float *lse, void *workspace, vsa_stream_t stream);

/* Forward straight from a block map, compacted inside the kernel (no LUT is built in
 * memory).
 *   block_map    int8, nonzero = attend.  map_shared == 0: [B, Hq, Sq/block, Sk/block],
 *                one map per (batch, query head); map_shared != 0: [Sq/block, Sk/block],
 *                one map for every batch and head (the Jenga layout).
 *   variable_block_sizes  [Sk/block] int32 valid keys per key block, or NULL = full.
 *   Shapes, lse, workspace and errors as vsa_fwd_gqa.  The result equals vsa_fwd_gqa on
 *   the LUT that vsa_bitmap_to_lut makes from the same map with max_kv = Sk/block.
 * Source: "FastVideo block_sparse_attn_sm100a.py", _block_sparse_attn_sm100a_from_mask_
 * inference and block_sparse_attn_sm100a_from_mask (a bool block_map [B, H, nb, nb] turned
 * into the forward's selection); "TheRock rocke sparse_attention.py", Jenga bullet of the
 * module docstring (an i8 map, nonzero = attend). */
VSA_API vsa_status vsa_fwd_from_mask(const vsa_bf16 *q, const vsa_bf16 *k, const vsa_bf16 *v,
                                     const int8_t *block_map, int map_shared,
                                     const int32_t *variable_block_sizes, int B, int Hq,
                                     int Hkv, int Sq, int Sk, int D, int block, float scale,
                                     vsa_bf16 *out, float *lse, void *workspace,
                                     vsa_stream_t stream);

/* Split-KV forward: vsa_fwd_gqa with each work item's key tiles divided into num_splits
 * contiguous ranges processed by different CTAs, then combined by a second kernel.  For
 * shapes with few work items (a short query, few heads) and long key lists, where one
 * CTA per item would leave most SMs idle.
 *   A work item is 128 query rows (one block-128 query block, or an adjacent pair of
 *   block-64 query blocks); its selected key blocks form key tiles of 128 keys, and range
 *   s of n tiles is tiles [n*s/num_splits, n*(s+1)/num_splits) (possibly empty).
 *   Each range leaves in the workspace an fp32 partial: O [128][128] relative to the
 *   row's running maximum m, then m, the sum of the bf16-rounded weights and the sum of
 *   the fp32 weights per row; the merge takes M = max m_s and c_s = 2^(m_s - M) and
 *   writes out = sum c_s O_s / sum c_s l_round_s and lse = M + log2(sum c_s l_exact_s),
 *   the same arithmetic the single-pass kernel uses to join its two key halves, so the
 *   result matches vsa_fwd_gqa within rounding (not bit for bit).
 *   num_splits   1..VSA_MAX_SPLITS; 1 is vsa_fwd_gqa (workspace then optional, as there).
 *   workspace    device memory of at least vsa_split_workspace_bytes(B, Hq, Sq, block,
 *                num_splits) bytes, 16-byte aligned, whose first vsa_workspace_bytes()
 *                bytes are zero before the call (they are left zero); the rest needs no
 *                initialisation.  Must not overlap q, out or lse.  Calls sharing a
 *                workspace must not overlap on the GPU.
 *   workspace_bytes  its size; a smaller one is VSA_ERR_INVALID_ARG.
 *   Other arguments and errors as vsa_fwd_gqa.  Enqueues two kernels.
 * Source: the split-K decode pattern of "vLLM FlyDSL tq_decode" (partial (m, l, O) per
 * key partition plus a reduction); the arithmetic of each part is that of vsa_fwd. */
VSA_API vsa_status vsa_fwd_split(const vsa_bf16 *q, const vsa_bf16 *k, const vsa_bf16 *v,
                                 const int32_t *q2k_idx, const int32_t *q2k_num,
                                 const int32_t *variable_block_sizes, int B, int Hq, int Hkv,
                                 int Sq, int Sk, int D, int max_kv, int block, float scale,
                                 int num_splits, vsa_bf16 *out, float *lse, void *workspace,
                                 size_t workspace_bytes, vsa_stream_t stream);

/* Workspace bytes vsa_fwd_split needs for this shape (0 for an invalid one). */
VSA_API size_t vsa_split_workspace_bytes(int B, int Hq, int Sq, int block, int num_splits);

/* Backward: dq, dk, dv of the vsa_fwd_gqa forward for an upstream gradient dout.
 *   With p_ij = 2^(scale * log2(e) * q_i . k_j - lse_i) over the attended keys (0 for the
 *   rest), D_i = dout_i . out_i and ds_ij = p_ij (dout_i . v_j - D_i):
 *     dq_i = scale sum_j ds_ij k_j,  dk_j = scale sum_i ds_ij q_i,  dv_j = sum_i p_ij dout_i,
 *   dk and dv summed over every query head of a key/value group.  Rows with no attended
 *   key contribute nothing (their dq is 0); keys no row attends get dk = dv = 0.
 *   q, k, v, q2k_idx, q2k_num, variable_block_sizes, shapes, max_kv, block, scale: as given
 *     to the forward.
 *   out          the forward's output [B, Hq, Sq, D] bf16.
 *   lse          the forward's lse [B, Hq, Sq] fp32 (required, 16-byte aligned).
 *   dout         [B, Hq, Sq, D] bf16.
 *   dq           [B, Hq, Sq, D] bf16 output;  dk, dv  [B, Hkv, Sk, D] bf16 outputs.
 *   workspace    at least vsa_bwd_workspace_bytes(B, Hq, Sq, Sk, block) bytes, 256-byte
 *                aligned, no initialisation needed (the block map, -D and -lse per
 *                query row and an fp32 dq accumulator live there).
 *   No output may overlap an input or another output.  Enqueues up to four kernels and
 *   one memset; errors as vsa_fwd_gqa, and VSA_ERR_UNSUPPORTED for more than 65536 query
 *   blocks per head or more than 4096 query heads per key/value head.
 * Source: "FastVideo block_sparse_attn_sm100a.py", module docstring (the backward
 * consumes the forward's base-2 lse); the gradient is that of softmax attention. */
VSA_API vsa_status vsa_bwd(const vsa_bf16 *q, const vsa_bf16 *k, const vsa_bf16 *v,
                           const vsa_bf16 *out, const vsa_bf16 *dout, const float *lse,
                           const int32_t *q2k_idx, const int32_t *q2k_num,
                           const int32_t *variable_block_sizes, int B, int Hq, int Hkv, int Sq,
                           int Sk, int D, int max_kv, int block, float scale, vsa_bf16 *dq,
                           vsa_bf16 *dk, vsa_bf16 *dv, void *workspace, size_t workspace_bytes,
                           vsa_stream_t stream);

/* Workspace bytes vsa_bwd needs for this shape (0 for an invalid one). */
VSA_API size_t vsa_bwd_workspace_bytes(int B, int Hq, int Sq, int Sk, int block);

/* Bytes of device workspace the forward entry points use when given one. */
VSA_API size_t vsa_workspace_bytes(void);

/* Size of the library's own scheduling scratch used by vsa_fwd_noalloc. */
#define VSA_NOALLOC_SCRATCH_BYTES 256

/* vsa_fwd for callers that cannot allocate device memory.  (The pages describe no such
 * entry point; it exists for this library's users.)  Some callers have no way to obtain
 * a workspace buffer: a plug-in whose host framework owns every device allocation and
 * offers no hook for extra buffers, or a serving loop that must not call cudaMalloc once
 * it is running because cudaMalloc can synchronise the device and stall other streams.
 * This entry point takes the same arguments as vsa_fwd minus `workspace`, allocates
 * nothing and calls no allocating routine: its dynamic-schedule scratch is a static
 * device array of VSA_NOALLOC_SCRATCH_BYTES bytes inside the library, which every GPU
 * that loads the library keeps until the process exits.
 *   - The first call on a device (with that device current) looks up the array's
 *     device address and caches it for the device's current context; a later call in
 *     a new context (after cudaDeviceReset, say) looks it up again.  Make the first
 *     call on a device before any stream capture begins.
 *   - Every call on a device shares the array, which keeps what the last call left.
 *     Each call clears the scheduling counters in stream order before its kernel, so
 *     calls on one stream are safe; calls that overlap on the GPU (different streams
 *     without ordering between them) race on the counters and must not be issued.
 *   - A call whose scratch need exceeds VSA_NOALLOC_SCRATCH_BYTES returns
 *     VSA_ERR_UNSUPPORTED.  Argument errors and unsupported configurations are those
 *     of vsa_fwd and are reported before anything is enqueued; a VSA_ERR_CUDA from a
 *     failed launch can come after the scratch reset was enqueued (harmless: the
 *     scratch is left zero). */
VSA_API vsa_status vsa_fwd_noalloc(const vsa_bf16 *q, const vsa_bf16 *k, const vsa_bf16 *v,
                                   const int32_t *q2k_idx, const int32_t *q2k_num,
                                   const int32_t *variable_block_sizes, int B, int H, int S,
                                   int D, int max_kv, int block, float scale, vsa_bf16 *out,
                                   float *lse, vsa_stream_t stream);

/* LUT -> bitmap, bit-exact: bitmap[r, kb] = 1 iff kb is one of the first
 * clamp(q2k_num[r], 0, max_kv) entries of q2k_idx row r (entries outside [0, nb)
 * skipped), else 0.  q2k_idx [rows, max_kv], q2k_num [rows], bitmap [rows, nb] int8.
 * Source: "TheRock rocke sparse_attention.py", _stage_vsa_bitmap_to_lds (zero the
 * row, then scatter 1 at every listed block; idempotent). */
VSA_API vsa_status vsa_lut_to_bitmap(const int32_t *q2k_idx, const int32_t *q2k_num, int rows,
                             int max_kv, int nb, int8_t *bitmap, vsa_stream_t stream);

/* bitmap -> LUT, bit-exact: row r lists the indices of its nonzero bytes in
 * ascending order, the first min(count, max_kv) of them, then -1 up to max_kv;
 * q2k_num[r] = min(count, max_kv).  bitmap [rows, nb] int8 -> q2k_idx [rows, max_kv],
 * q2k_num [rows] int32.
 * Source: "FastVideo block_sparse_attn_sm100a.py", _block_sparse_attn_sm100a_from_
 * mask_inference (a bool block map compacted into (q2k_idx, q2k_num), -1 fill). */
VSA_API vsa_status vsa_bitmap_to_lut(const int8_t *bitmap, int rows, int nb, int max_kv,
                             int32_t *q2k_idx, int32_t *q2k_num, vsa_stream_t stream);

/* vsa_fwd with HOST buffers: copies q, k, v, q2k_idx, q2k_num, variable_block_sizes
 * from host memory into the caller's device buffers (the d_* arguments, same shapes as
 * vsa_fwd), runs the forward, and copies out (and lse, if h_lse is not NULL) back to host
 * memory.  The work is split into chunks of consecutive (b, h) heads (about 20 MB of q,
 * k, v each, at most 32, at most one per head): a chunk's inputs go over on an input
 * stream, its forward runs on `stream` as soon as they have landed, and its outputs come
 * back on an output stream, so copies of one chunk overlap the forward of another.  The two internal streams (and their events) are created once
 * per device on first use -- no device memory -- and fork from `stream` at the start of
 * the call and join it at the end: everything is ordered after earlier work on `stream`,
 * and later work on `stream` (or a synchronisation of it) sees the whole call complete.
 * The caller synchronises `stream` before reading h_out / h_lse.  Host buffers should
 * be pinned (page-locked) for the copies to be asynchronous.  d_lse may be NULL only if
 * h_lse is NULL.  Calls from several host threads are serialised on an internal lock.
 * Argument errors are reported before anything is enqueued. */
VSA_API vsa_status vsa_fwd_from_host(const vsa_bf16 *h_q, const vsa_bf16 *h_k, const vsa_bf16 *h_v,
                             const int32_t *h_q2k_idx, const int32_t *h_q2k_num,
                             const int32_t *h_variable_block_sizes, int B, int H, int S,
                             int D, int max_kv, int block, float scale, vsa_bf16 *h_out,
                             float *h_lse, vsa_bf16 *d_q, vsa_bf16 *d_k, vsa_bf16 *d_v,
                             int32_t *d_q2k_idx, int32_t *d_q2k_num,
                             int32_t *d_variable_block_sizes, vsa_bf16 *d_out, float *d_lse,
                             void *workspace, vsa_stream_t stream);

/* Synchronises `stream`, then reads and clears the device status word of the current
 * device: VSA_OK, or VSA_ERR_DEVICE_TIMEOUT if a kernel gave up on a wait since the
 * last call (`detail`, if not NULL, receives the recorded code). */
VSA_API vsa_status vsa_device_status(vsa_stream_t stream, unsigned int *detail);

/* Number of kernel launches the most recent successful forward call on this thread
 * enqueued (for accounting in benchmarks). */
VSA_API int vsa_last_launch_count(void);

/* Test hooks for the timeout path (failure detection without a GPU fault).  Both are
 * process-wide settings read when a forward or backward kernel is launched; they change
 * no result of a launch that completes.  (The pages have no counterpart.)
 *   vsa_set_wait_limit_ns(ns): the limit of every internal wait that is not a drain
 *     (a drain waits for the kernel's own copies and MMAs in flight and always keeps the
 *     full limit of about one second, so nothing is in flight when a CTA exits).
 *     0 restores the full limit.  A short limit makes waits run out on ordinary work.
 *   vsa_set_stall_test(enable): while nonzero, the MMA warp of every CTA first waits on
 *     a barrier that nothing ever completes; that wait runs out after the limit above,
 *     records its code in the device status word (forward 0x11f, backward 0x15f), and
 *     every role of the CTA returns.  The launch's outputs are then undefined and
 *     vsa_device_status() reports VSA_ERR_DEVICE_TIMEOUT. */
VSA_API void vsa_set_wait_limit_ns(unsigned long long ns);
VSA_API void vsa_set_stall_test(int enable);

/* Static text for a status code. */
VSA_API const char *vsa_status_str(vsa_status s);

#ifdef __cplusplus
}
#endif

#endif /* VSA_GB300_H */
