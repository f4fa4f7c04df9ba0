/*
 * mcs.h — C ABI of libmcs: the MC-Sparse hot path on one NVIDIA GB300 (sm_103a).
 *
 * The operations follow the method described in "MC-Sparse: Deconstructing and
 * Closing the Dense-Sparse Attention Gap in Diffusion Transformers" (summary
 * page of arXiv 2610.06801). Paragraphs are cited by subject:
 *   [grouping]  index gathering and PDDP: queries are cut into groups of exactly
 *               C (the tile width) by projecting onto the principal direction,
 *               splitting at the median and repeating; keys and values are
 *               gathered from per-group index lists, not repacked into blocks;
 *   [selection] the anchor step's two-pass exact top-K: per group, the K keys
 *               with the largest summed attention weight; pass 1 is the row
 *               max / log-sum-exp, pass 2 recomputes the probabilities;
 *   [residual]  the anchor stores dense output minus sparse output; reuse steps
 *               add it to a fresh sparse attention of the current Q, K, V;
 *   [dense]     every anchor still runs full dense attention.
 *
 * Conventions shared by every entry point
 *   - Tensors q, k, v, o, residual are contiguous [B, H, N, d] with d fastest
 *     (row-major, one row per token), element type given by mcs_desc.dtype.
 *     N is the number of real tokens; N_pad = G*C with G = ceil(N/C) groups.
 *   - perm is int32 [B, H, N_pad]: for each (b, h), token ids listed group by
 *     group (group g occupies perm[g*C .. g*C+C-1]), ascending inside a group.
 *     Entries >= N are pad slots (zero queries; their outputs are never written).
 *   - group_of is int32 [B, H, N]: the group id of each real token.
 *   - idx is int32 [B, H, G, K]: per group, K key ids in [0, N), ascending.
 *   - lse is fp32 [B, H, N]: natural-log row log-sum-exp of the scaled logits.
 *   - Every pointer is a DEVICE pointer unless stated otherwise, owned by the
 *     caller, 16-byte aligned, and must stay valid until the stream reaches the
 *     call. Inputs may not alias outputs.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream). Argument errors are returned before anything is launched.
 *     A failed launch returns MCS_ERR_CUDA. Faults detected on the device (an
 *     index out of range) do not stop the kernel: the offending row is skipped,
 *     a sticky flag is raised, and mcs_check_status() reports it.
 *   - The library allocates no device memory except one small static word of
 *     device status flags and the fixed 64 MiB static score array of
 *     mcs_anchor_select_noalloc; all other scratch space is the caller's
 *     workspace. (mcs_sparse_attn_gather_host and the meta-cache ring create
 *     CUDA streams and events, no memory.)
 *   - No C++ exception crosses this boundary.
 */
#ifndef MCS_H_
#define MCS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *mcs_stream; /* same type as cudaStream_t */

typedef enum {
  MCS_OK = 0,
  MCS_ERR_INVALID_ARG = 1,    /* null/misaligned pointer, bad size, K out of [1, N] */
  MCS_ERR_UNSUPPORTED = 2,    /* d, C or dtype outside the supported set, or (mcs_anchor_select_noalloc)
                                 N too large for one score row in its fixed array */
  MCS_ERR_WORKSPACE = 3,      /* workspace pointer null or smaller than mcs_workspace_size() */
  MCS_ERR_CUDA = 4,           /* a CUDA runtime call or kernel launch failed */
  MCS_ERR_DEVICE_BOUNDS = 5,  /* a kernel met an index outside [0, N) (reported by mcs_check_status) */
  MCS_ERR_DEVICE_TIMEOUT = 6  /* a kernel's bounded wait ran out and it stopped early */
} mcs_status;

typedef enum { MCS_F32 = 0, MCS_BF16 = 1 } mcs_dtype;

/* Problem description. Supported: d in {64, 128}; C in {64, 128}; dtype F32 or
 * BF16 (BF16 runs on the tcgen05 tensor cores with fp32 accumulation, F32 runs
 * in fp32 SIMT arithmetic); B*H*N_pad < 2^31. scale <= 0 selects 1/sqrt(d).
 * pddp_iters <= 0 selects 20 power iterations. */
typedef struct {
  int B, H, N, d, C;
  int dtype;       /* mcs_dtype */
  float scale;
  int pddp_iters;
} mcs_desc;

/* Bytes of device workspace that mcs_group_pddp and mcs_anchor_select need for
 * this problem and this K (the larger of the two). Returns 0 for an invalid
 * description. Host-only; launches nothing. */
size_t mcs_workspace_size(const mcs_desc *desc, int K);

/* [grouping] PDDP grouping of each head's queries into G groups of exactly C.
 * Per (b, h) and per tree node of n >= 2 groups: mean of the node's real
 * queries, principal direction of the centred node by exactly pddp_iters power
 * iterations from 1/sqrt(d)*ones, projection of each member, and a rank split
 * sending the floor(n/2)*C members with the lowest (projection, token id) left.
 * Pads (ids >= N) sort last. Group ids are the depth-first leaf order.
 * q: [B,H,N,d]. Writes perm [B,H,N_pad] and group_of [B,H,N].
 * ws/ws_bytes: caller-owned device scratch, at least mcs_workspace_size(desc, 1)
 * bytes; its contents on entry are ignored. */
mcs_status mcs_group_pddp(const mcs_desc *desc, const void *q, int32_t *perm, int32_t *group_of,
                          void *ws, size_t ws_bytes, mcs_stream stream);

/* [grouping] "Fast PDDP": the same grouping with the power iteration of every
 * tree node started from a stored direction instead of 1/sqrt(d)*ones. The
 * pages report the grouping's cost amortised over the denoising steps without
 * describing how; this is the plainest reading: an anchor starts each node from
 * the direction the previous anchor found for it (the queries drift little
 * between anchors), so a few iterations (desc->pddp_iters, e.g. 4) do the work
 * of 20 from the fixed start.
 * Direction tables are fp32 [B, H, S, d] with S = 2^ceil(log2 G) - 1 rows per
 * head: tree node k of level l (root: level 0; the children of node k are
 * nodes 2k and 2k+1 of the next level) is row 2^l - 1 + k; rows of nodes that
 * do not split are unused. mcs_pddp_dirs_size() gives the bytes of one table
 * (0 for an invalid description). dirs_in: start directions or NULL (then
 * 1/sqrt(d)*ones, i.e. mcs_group_pddp); dirs_out: receives every split node's
 * final direction, or NULL; the two may be the same buffer. Iterations:
 * desc->pddp_iters when > 0; 0 with dirs_in given uses the stored directions
 * as they are; otherwise 20. Other arguments and results as mcs_group_pddp. */
size_t mcs_pddp_dirs_size(const mcs_desc *desc);
mcs_status mcs_group_pddp_warm(const mcs_desc *desc, const void *q, const float *dirs_in, float *dirs_out,
                               int32_t *perm, int32_t *group_of, void *ws, size_t ws_bytes, mcs_stream stream);

/* [dense] + [selection] pass 1: full softmax attention of every query over every
 * key, o_i = sum_j softmax_j(scale q_i.k_j) v_j, and the row log-sum-exp.
 * q, k, v: [B,H,N,d] inputs; o: [B,H,N,d] output (may be NULL to compute only
 * lse); lse: fp32 [B,H,N] output (may be NULL). At least one must be non-NULL. */
mcs_status mcs_dense_attn(const mcs_desc *desc, const void *q, const void *k, const void *v,
                          void *o, float *lse, mcs_stream stream);

/* [selection] pass 2 + exact top-K. For every group g: S_g[j] = sum over the
 * group's real queries i of exp(scale q_i.k_j - lse_i); idx[g] = the K keys with
 * the largest S_g (ties to the lower key id), written ascending.
 * perm: [B,H,N_pad] from mcs_group_pddp. lse: fp32 [B,H,N] from
 * mcs_dense_attn, or NULL to have pass 1 computed here (into the workspace).
 * idx: int32 [B,H,G,K] output. mass: fp32 [B,H,G] output or NULL; mass[g] =
 * sum_{j in idx[g]} S_g[j] / (real queries in g). ws: at least
 * mcs_workspace_size(desc, K) bytes. */
mcs_status mcs_anchor_select(const mcs_desc *desc, const void *q, const void *k, const int32_t *perm,
                             const float *lse, int K, int32_t *idx, float *mass,
                             void *ws, size_t ws_bytes, mcs_stream stream);

/* Anchor selection for callers that cannot allocate device memory (the method
 * has no counterpart: this is a deployment variant of mcs_anchor_select).
 * Code that runs where cudaMalloc is unavailable or forbidden (inside a
 * capture that must not allocate, a host framework that owns the device heap
 * and gives plug-ins no allocator, a loop that cannot afford cudaMalloc's
 * synchronisation) can call this instead: the pass-2 score rows live in one
 * fixed 64 MiB array inside the library (held by every GPU that loads it until
 * the process exits), so the call allocates nothing. Same arguments and results
 * as mcs_anchor_select, except that lse is required (pass 1 is not computed
 * here) and there is no workspace. Limits: N * 4 bytes (one score row) must fit
 * in the 64 MiB array, i.e. N <= 16,777,216, else MCS_ERR_UNSUPPORTED. The
 * first call on a device looks up the array's device address with that device
 * current; make that first call before any stream capture. All calls share the
 * array and leave their scores in it (nothing needs clearing: each call writes
 * every score it reads); calls whose kernels overlap on the GPU race on it. */
mcs_status mcs_anchor_select_noalloc(const mcs_desc *desc, const void *q, const void *k, const int32_t *perm,
                                     const float *lse, int K, int32_t *idx, float *mass, mcs_stream stream);

/* [grouping] + [residual] token-gather sparse attention. For every group g and
 * real member i: o_i = sum_{j in idx[g]} softmax_{idx[g]}(scale q_i.k_j) v_j
 * (renormalised over the kept keys), plus residual_i when residual != NULL.
 * Rows are read through perm and written back to their token positions; pad
 * slots are skipped. q, k, v: current-step [B,H,N,d]; idx: [B,H,G,K];
 * residual: [B,H,N,d] or NULL; o: [B,H,N,d] output. */
mcs_status mcs_sparse_attn_gather(const mcs_desc *desc, const void *q, const void *k, const void *v,
                                  const int32_t *perm, const int32_t *idx, int K,
                                  const void *residual, void *o, mcs_stream stream);

/* Host-to-host form of mcs_sparse_attn_gather for a reuse step whose current
 * q, k, v live in host memory and whose output is wanted there (the method has
 * no counterpart: this is a deployment variant). Same computation and result as
 * mcs_sparse_attn_gather, bit for bit. q_host, k_host, v_host: [B,H,N,d] host
 * buffers (pinned memory lets the copies overlap; pageable memory is correct
 * but serialises them); o_host: [B,H,N,d] host output; perm, idx, residual: the
 * meta-cache in device memory as for mcs_sparse_attn_gather. The B*H heads are
 * split into head_chunks chunks (at most one per head): chunk c is copied in on
 * a copy stream, computed on one of two internal streams (alternating, so that
 * consecutive chunks' kernels overlap at their edges), and copied out on a
 * second copy stream, so the copies of neighbouring chunks overlap the
 * kernels; two chunks are staged
 * in ws (device, 16-byte aligned, at least
 * mcs_sparse_attn_gather_host_workspace_size(desc, head_chunks) bytes). Work is
 * ordered after earlier work on `stream`, and `stream` is ordered after all of
 * it (synchronise `stream` before reading o_host). Errors: MCS_ERR_INVALID_ARG
 * for a bad argument, MCS_ERR_WORKSPACE for a small or misaligned ws,
 * MCS_ERR_CUDA if a stream, event or copy cannot be set up. */
size_t mcs_sparse_attn_gather_host_workspace_size(const mcs_desc *desc, int head_chunks);
mcs_status mcs_sparse_attn_gather_host(const mcs_desc *desc, const void *q_host, const void *k_host,
                                       const void *v_host, const int32_t *perm, const int32_t *idx, int K,
                                       const void *residual, void *o_host, void *ws, size_t ws_bytes,
                                       int head_chunks, mcs_stream stream);

/* Meta-cache ring: the per-layer cache {perm, idx, residual} of a model's
 * layers kept in HOST memory, with two device slots that take turns, so that a
 * layer's entry is copied in while the previous layer computes and a fresh
 * anchor entry is copied out while the next layer computes ([residual]: the
 * cache is reused across steps; holding it for every layer is what fills device
 * memory). All copies run on a stream the ring owns; compute on the caller's
 * stream is ordered against them with events, so nothing blocks the host.
 *
 * One entry is perm [B,H,N_pad] int32, idx [B,H,G,K] int32 and residual
 * [B,H,N,d] in the I/O dtype, each section 256-byte aligned, in
 * mcs_cache_entry_bytes(desc, K) bytes. host_entries: n_layers entries in host
 * memory (pinned for overlap), 256-byte aligned; device_slots: 2 entries in
 * device memory, 256-byte aligned; both owned by the caller and valid until
 * mcs_cache_ring_destroy returns. The ring is bound to the current device.
 *
 * mcs_cache_ring_acquire(layer, load, prefetch_next, stream, &perm, &idx,
 *   &residual): returns device pointers to the layer's slot. load = 1 makes
 *   the host entry resident first (nothing is copied when the slot already
 *   holds it, e.g. from a prefetch); load = 0 only reserves a slot, for an
 *   anchor step that will overwrite it. Work enqueued on `stream` afterwards
 *   sees the slot's contents. prefetch_next = 1 also starts copying layer
 *   (layer + 1) mod n_layers into the other slot, behind that slot's last
 *   release (skipped while the other slot is acquired or already holds it).
 *   At most two layers are acquired at once; a layer cannot be acquired twice.
 * mcs_cache_ring_release(layer, store, stream): the layer's kernels on
 *   `stream` are the last users of its slot; store = 1 then copies the slot
 *   back to the layer's host entry (after those kernels).
 * mcs_cache_ring_destroy: waits for the ring's copies, frees the ring.
 * Errors: MCS_ERR_INVALID_ARG for a bad argument or an acquire/release out of
 * order, MCS_ERR_CUDA if a stream, event or copy call fails. Calls on one ring
 * are serialised by a lock. */
typedef struct mcs_cache_ring_s *mcs_cache_ring;
size_t mcs_cache_entry_bytes(const mcs_desc *desc, int K);
mcs_status mcs_cache_ring_create(const mcs_desc *desc, int K, int n_layers, void *host_entries,
                                 void *device_slots, mcs_cache_ring *ring);
mcs_status mcs_cache_ring_acquire(mcs_cache_ring ring, int layer, int load, int prefetch_next,
                                  mcs_stream stream, int32_t **perm, int32_t **idx, void **residual);
mcs_status mcs_cache_ring_release(mcs_cache_ring ring, int layer, int store, mcs_stream stream);
mcs_status mcs_cache_ring_destroy(mcs_cache_ring ring);

/* [residual] anchor residual in one pass: the sparse attention of
 * mcs_sparse_attn_gather (without residual) is computed and r_i = o_dense_i -
 * o_sparse_i is written, in fp32 and rounded once to dtype. o_dense: [B,H,N,d]
 * from mcs_dense_attn; r: [B,H,N,d] output. */
mcs_status mcs_anchor_residual(const mcs_desc *desc, const void *q, const void *k, const void *v,
                               const int32_t *perm, const int32_t *idx, int K,
                               const void *o_dense, void *r, mcs_stream stream);

/* [residual] r = o_dense - o_sparse, element-wise over [B,H,N,d]. */
mcs_status mcs_residual_store(const mcs_desc *desc, const void *o_dense, const void *o_sparse, void *r,
                              mcs_stream stream);

/* [residual] o = o_sparse + r, element-wise over [B,H,N,d]. o may equal o_sparse. */
mcs_status mcs_residual_apply(const mcs_desc *desc, const void *o_sparse, const void *r, void *o,
                              mcs_stream stream);

/* Synchronises `stream`, then reports (and clears) the device-side flags raised
 * since the last call: MCS_ERR_DEVICE_BOUNDS, MCS_ERR_DEVICE_TIMEOUT, or a
 * sticky CUDA error as MCS_ERR_CUDA. MCS_OK if none. */
mcs_status mcs_check_status(mcs_stream stream);

/* Static, NUL-terminated description of a status code. Never NULL. */
const char *mcs_status_string(mcs_status status);

/* Number of kernels this process has launched through the library so far
 * (host-side counter, for launch accounting). */
uint64_t mcs_launch_count(void);

/* Diagnostic (no counterpart in the method): one tcgen05 MMA chain
 * D[128 x 128] = A[128 x 64] * B on the tensor cores, to check the shared-memory
 * descriptor encodings the attention kernels rely on. a: bf16 [128 x 64]
 * row-major; mode 0: b is bf16 [128 x 64] row-major (K-major operand,
 * D = A B^T); mode 1: b is bf16 [64 x 128] row-major (MN-major operand, D = A B)
 * with the descriptor's leading/stride byte offsets mn_lbo / mn_sbo; mode 2: as
 * mode 0 with A read from tensor memory. d: fp32 [128 x 128] output. All device
 * pointers. */
mcs_status mcs_selftest_tc_mma(const void *a, const void *b, float *d, int mode, uint32_t mn_lbo, uint32_t mn_sbo,
                               mcs_stream stream);

/* Diagnostic (no counterpart in the method): the failure path of the library's
 * bounded waits. Every pipeline wait inside the kernels (a stage that a copy or
 * an MMA should fill) gives up after a wall-time limit, raises the timeout flag,
 * lets its own copies land, frees its tensor memory and returns, instead of
 * hanging the GPU. This launches one CTA that holds tensor memory and waits on a
 * barrier nothing arrives at, with a limit of limit_ns (1 ns .. 10 s), so the
 * path can be exercised: afterwards mcs_check_status() returns
 * MCS_ERR_DEVICE_TIMEOUT (once) and the context stays usable. elapsed_ns: device
 * uint64 receiving the wait's duration in ns, or NULL. */
mcs_status mcs_selftest_wait_timeout(uint64_t limit_ns, uint64_t *elapsed_ns, mcs_stream stream);

/* Diagnostic (no counterpart in the method): the rate of the exponential unit as
 * the attention softmax uses it (ex2.approx.ftz.f32), which bounds kernels with
 * few FLOPs per exponential (d = 64 tiles, the pass-2 column sums). Launches
 * nblocks (1 .. 65535; one per SM gives the whole GPU) CTAs of 1,024 threads, one
 * per SM at a time, each thread running eight independent chains of `iters`
 * (1 .. 2^24) exponentials. out: device uint64 [nblocks][2] receiving each CTA's
 * duration in SM clock cycles and the number of exponentials it computed (their
 * ratio is exponentials per clock per SM). Asynchronous on `stream`. */
mcs_status mcs_selftest_ex2_rate(int iters, int nblocks, uint64_t *out, mcs_stream stream);

/* Diagnostic (no counterpart in the method): gathers 128 rows of the bf16 matrix
 * src [nrows x 128] (row-major, device) with TMA 4-row gathers into the swizzled
 * shared-memory layout of the attention kernels and writes them back row-major:
 * out[i, :] = src[rows[i], :], zeros where rows[i] >= nrows. rows: int32 [128]
 * device; out: bf16 [128 x 128] device. */
mcs_status mcs_selftest_tma_gather(const void *src, int nrows, const int32_t *rows, void *out, mcs_stream stream);

#ifdef __cplusplus
}
#endif
#endif /* MCS_H_ */
