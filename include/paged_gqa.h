/*
 * paged_gqa.h -- C ABI of the paged grouped-query decode attention library
 * (libpaged_gqa.so), sm_103a (GB300).
 *
 * The operation.  One decode step of attention: every sequence b of a batch
 * has one new query token with Hq heads, and Lb cached key/value tokens held
 * in a paged KV cache.  For each sequence b and query head h
 *
 *     kv      = h / G,   G = Hq / Hkv          (contiguous query-head groups)
 *     k_t,v_t = token t of sequence b, t in [0, Lb), stored in physical block
 *               block_table[b][t / block_size] at slot t % block_size
 *     out[b,h,:] = sum_t softmax_t(scale * <q[b,h,:], k_t>) v_t
 *
 * Sources: the attention equation Attention(Q,K,V) = softmax(Q K^T / sqrt(d)) V
 * ("Modern LLM Inference - Workloads, Bottlenecks, and Optimization
 * Techniques", section "Why Cross-Layer Attention Shares K/V but Not Q");
 * grouped-query attention, N query heads sharing K key/value heads (same notes,
 * section 4.1, and "The Ultimate Guide to LLM Inference Optimization - Part 2",
 * section "Grouped Query Attention": heads divisible by KV groups); the paged
 * cache, fixed-size blocks found through a block table ("Advanced
 * Optimizations: MQA, GQA, and PagedAttention", section "PagedAttention: The OS
 * Analogy"; "Modern LLM Inference ...", section 8.2 "Paged Attention";
 * "The Ultimate Guide ... Part 2", section "Paged Attention").  Reading the
 * block pages inside the attention kernel itself follows the "kernel fusion"
 * remark of "Modern LLM Inference ...", section 8.3.
 *
 * Layouts (all row-major, contiguous, device memory, 16-byte aligned):
 *     q            [B, Hq, D]                          dtype
 *     k_pool       [num_blocks, block_size, Hkv, D]    dtype
 *     v_pool       [num_blocks, block_size, Hkv, D]    dtype
 *     block_table  [B, max_blocks]                     int32
 *     seq_lens     [B]                                 int32
 *     out          [B, Hq, D]                          dtype
 * dtype is float32 or bfloat16 (PGD_F32 / PGD_BF16), or 8-bit pages (e4m3
 * floats or int8 integers, scaled per KV head or per block and KV head) with
 * bfloat16 q and out (PGD_FP8_E4M3 / PGD_INT8, paged_kv_pool_create_fp8 and
 * paged_kv_pool_create_q8); accumulation is float32.
 * D (head_dim) is 64 or 128; G = Hq / Hkv is 1..64; block_size is 1..256
 * (bfloat16 pools need a power of two in 8..256).
 *
 * Ownership.  The caller owns every buffer: the pools, q, the tables, out and
 * the workspace.  A pool handle is a non-owning, immutable description of the
 * two pool allocations; the library allocates only one 4-byte device error
 * word per handle (freed by paged_kv_pool_destroy).
 *
 * Errors.  Every call returns a pgd_status and never throws.  Argument errors
 * are returned before anything is launched.  paged_gqa_decode is asynchronous
 * on `stream`; faults the device finds (a block id outside [0, num_blocks), a
 * length outside [0, max_blocks * block_size], a pipeline wait that gave up)
 * are latched in the handle's error word and returned by paged_gqa_get_error.
 * The rows of an affected sequence are written as NaN.  The kernels never trap.
 *
 * Threads and streams.  A handle may be used from several host threads and
 * streams at once as long as concurrent decodes use distinct workspaces and
 * outputs.
 */
#ifndef PAGED_GQA_H
#define PAGED_GQA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pgd_pool_s *pgd_pool_t;

enum pgd_dtype { PGD_F32 = 0, PGD_BF16 = 1, PGD_FP8_E4M3 = 2, PGD_INT8 = 3 };

/* Granularity of the scales of 8-bit pages. */
enum pgd_scale_granularity {
    PGD_SCALE_PER_HEAD = 0,  /* k_scale / v_scale [Hkv] */
    PGD_SCALE_PER_BLOCK = 1  /* k_scale / v_scale [num_blocks, Hkv] */
};

enum pgd_status {
    PGD_OK = 0,
    PGD_ERR_ARG = 1,         /* null pointer, negative or zero size, bad enum value */
    PGD_ERR_SHAPE = 2,       /* Hq % Hkv != 0, unsupported head_dim / group / block size */
    PGD_ERR_DTYPE = 3,       /* unknown dtype */
    PGD_ERR_ALIGN = 4,       /* a pointer is not 16-byte aligned */
    PGD_ERR_WORKSPACE = 5,   /* workspace missing, misaligned or smaller than required */
    PGD_ERR_CUDA = 6,        /* a CUDA runtime or driver call failed */
    PGD_ERR_BLOCK_ID = 7,    /* device: a block id outside [0, num_blocks) (latched) */
    PGD_ERR_SEQ_LEN = 8,     /* device: a length outside [0, max_blocks*block_size] (latched) */
    PGD_ERR_UNSUPPORTED = 9, /* valid request this build does not implement */
    PGD_ERR_TIMEOUT = 10,    /* device: a pipeline wait gave up (latched) */
    PGD_ERR_TOO_LARGE = 11   /* paged_gqa_decode_noalloc: scratch need above its fixed size */
};

/*
 * Describe a K/V block pool pair resident on the current CUDA device.
 *   out          receives the handle (set to NULL on error)
 *   k_pool,
 *   v_pool       device pointers, [num_blocks, block_size, num_kv_heads, head_dim]
 *   num_blocks   physical blocks in each pool (>= 1)
 *   block_size   tokens per block
 *   num_kv_heads Hkv (>= 1)
 *   head_dim     D, 64 or 128
 *   dtype        PGD_F32 or PGD_BF16
 * The pools are not copied; they must outlive the handle.  Builds the TMA
 * descriptors the bfloat16 kernel walks the pool with.
 */
int paged_kv_pool_create(pgd_pool_t *out, const void *k_pool, const void *v_pool,
                         int64_t num_blocks, int block_size, int num_kv_heads, int head_dim,
                         int dtype);

/*
 * Describe a pool pair of 8-bit K/V pages: k_pool / v_pool hold e4m3 bytes
 * (1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, no infinities),
 * [num_blocks, block_size, num_kv_heads, 128]; element (block, slot, h, d)
 * stands for k_scale[h] * e4m3(byte) (v_scale[h] for V).  k_scale and
 * v_scale are device float32 arrays of num_kv_heads entries that must outlive
 * the handle.  Queries and outputs stay bfloat16 (q must be below 65504 in
 * magnitude: q . K is formed in f16).  block_size: a power of two in 8..256.
 * Quantized KV pages halve the bytes decode reads ("Modern LLM Inference ...",
 * section 6; "The Ultimate Guide ... Part 2", "KV Cache Compression").
 */
int paged_kv_pool_create_fp8(pgd_pool_t *out, const void *k_pool, const void *v_pool,
                             const float *k_scale, const float *v_scale, int64_t num_blocks,
                             int block_size, int num_kv_heads, int head_dim);

/*
 * Describe a pool pair of 8-bit K/V pages of either code, with scales of
 * either granularity.
 *   code         PGD_FP8_E4M3 (e4m3 bytes, as for paged_kv_pool_create_fp8) or
 *                PGD_INT8 (two's-complement integers in [-128, 127])
 *   granularity  PGD_SCALE_PER_HEAD: k_scale / v_scale are [num_kv_heads];
 *                element (block, slot, h, d) stands for k_scale[h] * code.
 *                PGD_SCALE_PER_BLOCK: k_scale / v_scale are [num_blocks,
 *                num_kv_heads] (row-major); element (block, slot, h, d)
 *                stands for k_scale[block * num_kv_heads + h] * code, so each
 *                physical block carries its own range (a cache written token
 *                by token fixes a block's scale when it writes the block).
 * The other arguments and rules are those of paged_kv_pool_create_fp8
 * (head_dim 128, block_size a power of two in 8..256, bfloat16 q and out).
 * The scale arrays are read by the decode kernels at every call, so a caller
 * may rewrite a block's row between calls (stream-ordered).  Quantized KV
 * pages: int8 / fp8 quantization, "Modern LLM Inference ...", section 6;
 * "The Ultimate Guide ... Part 2", "KV Cache Compression".
 * PGD_ERR_DTYPE for another code, PGD_ERR_ARG for another granularity or a
 * null scale array.
 */
int paged_kv_pool_create_q8(pgd_pool_t *out, const void *k_pool, const void *v_pool, int code,
                            const float *k_scale, const float *v_scale, int granularity,
                            int64_t num_blocks, int block_size, int num_kv_heads, int head_dim);

/* Release a handle (not the pools).  NULL is accepted. */
int paged_kv_pool_destroy(pgd_pool_t pool);

/*
 * Workspace bytes paged_gqa_decode needs for B sequences, Hq query heads and
 * `num_splits` (same meaning as in paged_gqa_decode; 0 = automatic).  Written
 * to *bytes.  The workspace holds per-split partial results, the tile prefix
 * table and one counter word per split run.  It must be zero-filled before
 * its first use; every call that completes leaves it ready for the next one
 * (each run's count back at zero; a flag bit beside it alternates), so a
 * workspace can be reused call after call.  After a call that latched
 * PGD_ERR_TIMEOUT, zero it again.
 */
int paged_gqa_workspace_size(pgd_pool_t pool, int B, int Hq, int num_splits, size_t *bytes);

/*
 * Enqueue one decode step on `stream` (a cudaStream_t; NULL = legacy default
 * stream).
 *   q, out       [B, Hq, D] in the pool's dtype (bfloat16 for 8-bit pools); out
 *                may not alias q
 *   block_table  [B, max_blocks] int32; entries past ceil(Lb / block_size) are
 *                never read and may hold anything
 *   seq_lens     [B] int32, cached tokens per sequence; Lb == 0 gives zeros
 *   scale        logit scale, usually 1/sqrt(D)
 *   workspace    device buffer of at least paged_gqa_workspace_size bytes,
 *                256-byte aligned, zero-filled before first use (see above);
 *                calls that may overlap on the GPU need distinct workspaces
 *   num_splits   how many equal spans the total KV work (all sequences times
 *                KV heads, in tiles of 16 tokens for 8 KV heads at a time with
 *                bfloat16 pages, 32 with 8-bit pages, 64 tokens of one head with
 *                float32) is cut into, one CTA each; a sequence crossing a span
 *                boundary is finished by a log-sum-exp merge.  0 = automatic
 *                (one span per SM, at least two tiles per span).
 * The result does not depend on num_splits beyond float32 rounding.
 * One kernel launch per call (two for float32 pools).  When the splits leave
 * long runs to merge and the grid fits on the device at once, the launch is
 * cooperative (the CTAs that share a run merge it together); if the driver
 * refuses that, the ordinary launch is used.
 */
int paged_gqa_decode(pgd_pool_t pool, const void *q, int B, int Hq, const int32_t *block_table,
                     int max_blocks, const int32_t *seq_lens, float scale, void *out,
                     void *workspace, size_t workspace_bytes, int num_splits, void *stream);

/*
 * Decode with several query tokens per sequence and an optional attention
 * window: speculative verification of drafted tokens ("Modern LLM Inference
 * ...", section 7.1) and local attention over the most recent tokens (same
 * notes, section 4.4 "Local Attention").
 *   q, out       [B, q_len, Hq, D], bfloat16 pools only (PGD_ERR_UNSUPPORTED
 *                for float32 with q_len > 1 or window > 0)
 *   seq_lens     cached tokens per sequence, the q_len query tokens included:
 *                they are the last q_len, already appended.  Query i sits at
 *                position p = Lb - q_len + i and attends causally to positions
 *                [lo, p], lo = max(0, p - window + 1) when window > 0, else 0.
 *                A query with p < 0 gets zeros.
 *   window       0 = no window.  Blocks that lie wholly before every query's
 *                window are never read, so their table entries may be -1.
 * q_len * Hq / Hkv must be at most 64.  The workspace size comes from
 * paged_gqa_workspace_size_ex.  q_len = 1 with window = 0 is paged_gqa_decode.
 */
int paged_gqa_decode_ex(pgd_pool_t pool, const void *q, int B, int q_len, int Hq,
                        const int32_t *block_table, int max_blocks, const int32_t *seq_lens,
                        int window, float scale, void *out, void *workspace,
                        size_t workspace_bytes, int num_splits, void *stream);

/* Workspace bytes for paged_gqa_decode_ex with q_len query tokens. */
int paged_gqa_workspace_size_ex(pgd_pool_t pool, int B, int q_len, int Hq, int num_splits,
                                size_t *bytes);

/*
 * Synchronise `stream`, then read and clear the handle's latched device error.
 * Returns PGD_OK when no error was latched, the latched pgd_status otherwise,
 * or PGD_ERR_CUDA when the synchronisation itself failed.
 */
int paged_gqa_get_error(pgd_pool_t pool, void *stream);

/* Number of spans num_splits = 0 resolves to for this handle's device. */
int paged_gqa_auto_splits(pgd_pool_t pool, int *num_splits);

/* Static, human-readable name of a pgd_status. */
const char *paged_gqa_strerror(int status);

/*
 * paged_gqa_decode without a workspace argument, for callers that cannot
 * allocate device memory: a plugin inside a host runtime that owns all device
 * memory and offers it no allocator, or a latency-critical path that must not
 * call cudaMalloc / cudaFree because they can synchronise the device.  (The
 * pages describe no such entry point; it is a property of this library.)
 *
 * Same arguments, semantics and errors as paged_gqa_decode, minus workspace.
 * The split-KV scratch is a fixed array of paged_gqa_noalloc_scratch_bytes()
 * bytes (16 MiB) of static device memory in this library, reserved on every
 * device that loads it until the process exits.  Requests whose workspace
 * (paged_gqa_workspace_size) exceeds that return PGD_ERR_TOO_LARGE before
 * anything is enqueued, and so does every argument error (with the status
 * paged_gqa_decode gives it): a refused call never touches the array.
 * Nothing is allocated: the first call on a device
 * looks up the array's device address with that device made current (make
 * that first call before any stream capture), and every call clears the
 * array's counters with cudaMemsetAsync on `stream` before the kernel.
 * All calls share the one array: calls that may overlap on the GPU (on
 * different streams, or from several threads) race on it and must be
 * serialised by the caller.
 */
int paged_gqa_decode_noalloc(pgd_pool_t pool, const void *q, int B, int Hq,
                             const int32_t *block_table, int max_blocks, const int32_t *seq_lens,
                             float scale, void *out, int num_splits, void *stream);

/* Size in bytes of the fixed scratch array paged_gqa_decode_noalloc uses. */
size_t paged_gqa_noalloc_scratch_bytes(void);

/*
 * paged_gqa_decode_ex with the step's inputs (q, block_table, seq_lens) and
 * its output in HOST memory; the pools stay in device memory.  (The pages
 * describe no such entry point; it is a property of this library.)
 *
 * Each of the four host buffers that is page-locked (cudaHostAlloc /
 * cudaMallocHost / cudaHostRegister, so mapped into the device's address
 * space) and aligned as paged_gqa_decode_ex requires (16 bytes for q and out,
 * 4 for the int32 arrays) is read or written by the kernel itself through its
 * mapped address, over the host link; every other buffer is staged through
 * the workspace with cudaMemcpyAsync on `stream` (for pageable memory that
 * copy may block the calling thread).  Either way the call is ordered on
 * `stream`, and h_out holds the result once the stream has synchronised; the
 * inputs must stay unchanged until then.  When h_out is written in place, the
 * split runs are merged inside the decode kernel (plan merge 0 where
 * paged_gqa_plan reports 2), so that only one kernel writes over the link.
 *   workspace    device buffer of at least paged_gqa_workspace_size_host
 *                bytes, 256-byte aligned; its first
 *                paged_gqa_workspace_size_ex bytes are the decode workspace
 *                (zero-filled before first use, reusable as described there),
 *                the rest is staging room for q, block_table, seq_lens and out
 * Arguments, shapes, results and errors otherwise as paged_gqa_decode_ex.
 * Returns PGD_ERR_CUDA if a staging copy cannot be enqueued.
 */
int paged_gqa_decode_host(pgd_pool_t pool, const void *h_q, int B, int q_len, int Hq,
                          const int32_t *h_block_table, int max_blocks,
                          const int32_t *h_seq_lens, int window, float scale, void *h_out,
                          void *workspace, size_t workspace_bytes, int num_splits, void *stream);

/*
 * The launch plan paged_gqa_decode_ex would use for these shapes, computed on
 * the host from the shapes alone (no device, no pool): dtype, num_kv_heads and
 * head_dim as for paged_kv_pool_create, num_sms the SM count of the device
 * (152 on GB300), the other arguments as for paged_gqa_decode_ex.  Writes five
 * ints to plan:
 *   plan[0]  KV heads per unit of work (the head group one tile covers)
 *   plan[1]  m16 row tiles of one KV head's q_len * Hq / Hkv query rows
 *   plan[2]  tokens per tile
 *   plan[3]  CTAs of the grid; with num_splits = 0 the kernel then uses
 *            min(plan[3], ceil(tiles / 2)) of them, tiles counted from the
 *            lengths on the device
 *   plan[4]  split merge: 0 by the warp whose piece completes a run, 1 shared
 *            among all the run's pieces under a cooperative launch (only
 *            when the grid, one CTA per SM, fits at once: plan[3] <= num_sms;
 *            should the device still refuse that launch, the library runs 0
 *            instead), 2 none in the decode kernel: its pieces only write
 *            partials and a second kernel merges every split run (runs over
 *            2 to 5 spans), 3 the float32 path's merge kernel
 * Returns the status paged_gqa_decode_ex returns for these shapes before any
 * pointer is looked at (PGD_ERR_SHAPE, PGD_ERR_UNSUPPORTED, ...).  A
 * diagnostic of this library; the pages have no counterpart.
 */
int paged_gqa_plan(int dtype, int num_kv_heads, int head_dim, int num_sms, int B, int q_len,
                   int Hq, int num_splits, int window, int *plan);

/* Workspace bytes for paged_gqa_decode_host (decode workspace + staging room). */
int paged_gqa_workspace_size_host(pgd_pool_t pool, int B, int q_len, int Hq, int max_blocks,
                                  int num_splits, size_t *bytes);

/*
 * Diagnostic of the failure path: launch one thread that waits, with the
 * bounded wait the pipeline kernels use and a limit of limit_us microseconds
 * (1 .. 1e6), on a barrier nothing arrives on.  The wait gives up, latches
 * PGD_ERR_TIMEOUT in the handle's error word (read it with
 * paged_gqa_get_error) and the kernel returns; nothing faults and the context
 * stays usable.  The pages have no counterpart; it tests this library.
 */
int paged_gqa_selftest_wait_timeout(pgd_pool_t pool, int64_t limit_us, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_GQA_H */
