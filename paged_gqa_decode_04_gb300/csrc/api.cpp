// C ABI of libpaged_gqa.so: argument checks, pool descriptors, workspace
// carve-up and kernel dispatch.  See include/paged_gqa.h for the contract.
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <new>

#include "paged_kv_manager.h"
#include "pgd_internal.h"

struct pgd_pool_s {
    pgd::Pool p;
};

namespace pgd {

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// 8-bit pages (either code)
bool is_q8(int dtype) { return dtype == PGD_FP8_E4M3 || dtype == PGD_INT8; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Make `dev` current for the scope of a call; restore the caller's device.
struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) {
            ok = false;
            return;
        }
        if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

PFN_cuTensorMapEncodeTiled_v12000 lookup_encode_fn() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return nullptr;
}

// The driver's tensor-map encoder, looked up once (a function-local static is
// initialised once even when several threads create pools together).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = lookup_encode_fn();
    return fn;
}

// 4-D view of a bf16 pool [num_blocks, bs, Hkv, D] listed as
// (d_lo = 64, slot = bs, head-half = Hkv*D/64, block = num_blocks), so that a
// box (64, rows, hg*D/64, 1) -- `rows` slots of one block for hg consecutive
// KV heads -- lands in shared memory head-half-major: [head-half][slot][64].
// 8-bit pages: the same view with one 128-byte row per head (D = 128 bytes):
// (d 128, slot, head, block), uint8 elements.
bool encode_pool_map(CUtensorMap* map, const void* base, int64_t num_blocks, int bs, int hkv,
                     int d, int hg, bool fp8) {
    auto fn = encode_fn();
    if (!fn) return false;
    const int elt = fp8 ? 1 : 2;
    const int row_elems = 128 / elt;                        // elements in a 128-byte row
    const int rows_per_head = d * elt / 128;                // 128-byte rows of one head
    const cuuint64_t row_bytes = (cuuint64_t)hkv * d * elt;  // one slot, all heads
    const int tile = (fp8 ? 256 : 128) / hg;  // tokens per tile of the decode kernel
    cuuint64_t dims[4] = {(cuuint64_t)row_elems, (cuuint64_t)bs,
                          (cuuint64_t)hkv * rows_per_head, (cuuint64_t)num_blocks};
    cuuint64_t strides[3] = {row_bytes, 128, row_bytes * bs};
    cuuint32_t box[4] = {(cuuint32_t)row_elems, (cuuint32_t)(bs < tile ? bs : tile),
                         (cuuint32_t)(hg * rows_per_head), 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                    4, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int resolve_parts(const Pool& p, int num_splits) {
    return num_splits > 0 ? num_splits : p.num_sms;
}

}  // namespace

const Pool& pool_desc(pgd_pool_t h) { return h->p; }

static int choose_hg_for(int dtype, int hkv, int rows) {
    if (dtype == PGD_F32) return 1;
    const int mt = (rows + 15) / 16;
    const int cap = mt == 1 ? 8 : mt == 2 ? 4 : 2;  // at most 8 consumer warps
    int hg = 8;
    while (hg > 1 && (hkv % hg != 0 || hg > cap)) hg /= 2;
    return hg;
}

int choose_hg(const Pool& p, int rows) { return choose_hg_for(p.dtype, p.hkv, rows); }

// The launch plan of a decode call, from shapes alone.  Status as the decode
// entry points return it for these shapes.
static int make_plan(int dtype, int hkv, int d, int num_sms, int B, int q_len, int Hq,
                     int num_splits, int window, Plan* out) {
    if (hkv < 1 || Hq < 1 || B < 0 || q_len < 1 || num_sms < 1 || num_splits < 0 ||
        num_splits > (1 << 20) || window < 0)
        return PGD_ERR_ARG;
    if (dtype != PGD_F32 && dtype != PGD_BF16 && !is_q8(dtype)) return PGD_ERR_DTYPE;
    if (d != 64 && d != 128) return PGD_ERR_SHAPE;
    if (is_q8(dtype) && d != 128) return PGD_ERR_SHAPE;
    if (Hq % hkv != 0) return PGD_ERR_SHAPE;
    const int rows = q_len * (Hq / hkv);
    if (rows > kMaxGroup) return PGD_ERR_SHAPE;
    if (dtype == PGD_F32 && (q_len > 1 || window > 0)) return PGD_ERR_UNSUPPORTED;
    Plan pl;
    pl.hg = choose_hg_for(dtype, hkv, rows);
    pl.m_tiles = (rows + 15) / 16;
    pl.tile_tokens = dtype == PGD_F32 ? kSimpleTileTokens : (is_q8(dtype) ? 256 : 128) / pl.hg;
    pl.parts = num_splits > 0 ? num_splits : num_sms;
    // Merge variant from the expected size of a split run's merge: about
    // parts / runs + 1 pieces per run, times the row passes of one warp.
    pl.merge_variant = dtype == PGD_F32 ? 3 : 0;
    if (dtype != PGD_F32 && d == 128 && B > 0) {
        const int runs = B * (hkv / pl.hg);
        const int nr = rows < 16 ? rows : 16;          // rows of one warp's m-tile
        const int passes = (nr * d + 127) / 128;       // 128 / D rows per merge pass
        const int64_t loads = (int64_t)passes * (pl.parts / runs + 1);
        if (nr >= 2 && loads > kShareMinLoads) pl.merge_variant = 1;
        else if (nr >= kSepMinRows && 2 * runs <= pl.parts && pl.parts <= 5 * runs &&
                 runs * pl.hg >= num_sms)
            pl.merge_variant = 2;
        // two or more row tiles per head: sharing each run's merge among its
        // pieces' warps beats one warp per row tile merging them all (measured)
        else if (pl.m_tiles >= 2)
            pl.merge_variant = 1;
        // the shared merge waits on other CTAs, so its grid must be resident
        // at once; the TMA kernel's shared memory (over half an SM's) allows
        // one CTA per SM, so a grid above the SM count takes the last arriver
        if (pl.merge_variant == 1 && pl.parts > num_sms) pl.merge_variant = 0;
    }
    *out = pl;
    return PGD_OK;
}

WorkspaceLayout workspace_layout(int B, int hkv, int rows_per_head, int hg, int d, int parts) {
    WorkspaceLayout w;
    const int mtiles = (rows_per_head + 15) / 16;
    const size_t rows = (size_t)hg * rows_per_head;  // rows of one partial result
    w.counters_off = 0;
    w.tile_base_off = round_up((size_t)B * hkv * mtiles * sizeof(int), 256);
    w.part_lse_off = w.tile_base_off + round_up((size_t)(B + 3) * sizeof(int64_t), 256);
    w.part_o_off = w.part_lse_off + round_up((size_t)parts * 2 * rows * sizeof(float), 256);
    w.total = w.part_o_off + round_up((size_t)parts * 2 * rows * d * sizeof(float), 256);
    return w;
}

int check_decode(const Pool& p, const void* q, int B, int q_len, int Hq,
                 const int32_t* block_table, int max_blocks, const int32_t* seq_lens, int window,
                 float scale, const void* out, const void* workspace, size_t workspace_bytes,
                 int num_splits, Plan* plan, WorkspaceLayout* wl) {
    if (B < 0 || q_len < 1 || Hq < 1 || max_blocks < 0 || num_splits < 0 ||
        num_splits > (1 << 20) || window < 0)
        return PGD_ERR_ARG;
    if (!isfinite(scale)) return PGD_ERR_ARG;
    {
        const int rc = make_plan(p.dtype, p.hkv, p.d, p.num_sms, B, q_len, Hq, num_splits,
                                 window, plan);
        if (rc != PGD_OK) return rc;
    }
    if ((int64_t)max_blocks * p.block_size > INT32_MAX) return PGD_ERR_SHAPE;
    if (B == 0) return PGD_OK;
    if (!q || !out || !block_table || !seq_lens || !workspace) return PGD_ERR_ARG;
    if (max_blocks < 1) return PGD_ERR_SHAPE;
    const size_t elt = p.dtype == PGD_F32 ? 4 : 2;  // q / out element (bf16 for 8-bit pages)
    const size_t qbytes = (size_t)B * q_len * Hq * p.d * elt;
    {
        const uintptr_t q0 = reinterpret_cast<uintptr_t>(q), o0 = reinterpret_cast<uintptr_t>(out);
        if (q0 < o0 + qbytes && o0 < q0 + qbytes) return PGD_ERR_ARG;  // out aliases q
    }
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(block_table, 4) ||
        !aligned(seq_lens, 4))
        return PGD_ERR_ALIGN;
    *wl = workspace_layout(B, p.hkv, q_len * (Hq / p.hkv), plan->hg, p.d, plan->parts);
    if (!aligned(workspace, 256) || workspace_bytes < wl->total) return PGD_ERR_WORKSPACE;
    return PGD_OK;
}

}  // namespace pgd

using namespace pgd;

extern "C" {

static int pool_create(pgd_pool_t* out, const void* k_pool, const void* v_pool,
                       const float* k_scale, const float* v_scale, int scale_per_block,
                       int64_t num_blocks, int block_size, int num_kv_heads, int head_dim,
                       int dtype) {
    if (!out) return PGD_ERR_ARG;
    *out = nullptr;
    if (!k_pool || !v_pool) return PGD_ERR_ARG;
    if (num_blocks < 1 || num_blocks > INT32_MAX || block_size < 1 || num_kv_heads < 1)
        return PGD_ERR_ARG;
    if (dtype != PGD_F32 && dtype != PGD_BF16 && !is_q8(dtype)) return PGD_ERR_DTYPE;
    if (head_dim != 64 && head_dim != 128) return PGD_ERR_SHAPE;
    if (block_size > 1024) return PGD_ERR_SHAPE;
    if (dtype != PGD_F32 &&
        (block_size < 8 || block_size > 256 || (block_size & (block_size - 1)) != 0))
        return PGD_ERR_SHAPE;
    if (is_q8(dtype)) {
        if (head_dim != 128) return PGD_ERR_SHAPE;
        if (!k_scale || !v_scale) return PGD_ERR_ARG;
        if (!aligned(k_scale, 4) || !aligned(v_scale, 4)) return PGD_ERR_ALIGN;
    }
    if (!aligned(k_pool, 16) || !aligned(v_pool, 16)) return PGD_ERR_ALIGN;

    pgd_pool_s* h = new (std::nothrow) pgd_pool_s;
    if (!h) return PGD_ERR_ARG;
    memset(h, 0, sizeof(*h));
    Pool& p = h->p;
    p.k = k_pool;
    p.v = v_pool;
    p.num_blocks = num_blocks;
    p.block_size = block_size;
    p.hkv = num_kv_heads;
    p.d = head_dim;
    p.dtype = dtype;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.scale_per_block = scale_per_block;
    if (cudaGetDevice(&p.device) != cudaSuccess || p.device >= kMaxDevices ||
        cudaDeviceGetAttribute(&p.num_sms, cudaDevAttrMultiProcessorCount, p.device) !=
            cudaSuccess ||
        cudaMalloc(reinterpret_cast<void**>(&p.err), sizeof(int)) != cudaSuccess) {
        delete h;
        return PGD_ERR_CUDA;
    }
    if (cudaMemset(p.err, 0, sizeof(int)) != cudaSuccess) {
        cudaFree(p.err);
        delete h;
        return PGD_ERR_CUDA;
    }
    if (dtype != PGD_F32) {
        const bool fp8 = is_q8(dtype);  // 8-bit pages of either code: uint8 tensor maps
        for (int i = 0; i < 4; ++i) {
            const int hg = 1 << i;
            if (num_kv_heads % hg != 0) continue;
            if (!encode_pool_map(&p.tmap_k[i], k_pool, num_blocks, block_size, num_kv_heads,
                                 head_dim, hg, fp8) ||
                !encode_pool_map(&p.tmap_v[i], v_pool, num_blocks, block_size, num_kv_heads,
                                 head_dim, hg, fp8)) {
                cudaFree(p.err);
                delete h;
                return PGD_ERR_CUDA;
            }
            p.tmap_ok[i] = true;
        }
    }
    *out = h;
    return PGD_OK;
}

int paged_kv_pool_create(pgd_pool_t* out, const void* k_pool, const void* v_pool,
                         int64_t num_blocks, int block_size, int num_kv_heads, int head_dim,
                         int dtype) {
    if (is_q8(dtype)) return PGD_ERR_ARG;  // needs scales: paged_kv_pool_create_q8
    return pool_create(out, k_pool, v_pool, nullptr, nullptr, 0, num_blocks, block_size,
                       num_kv_heads, head_dim, dtype);
}

int paged_kv_pool_create_fp8(pgd_pool_t* out, const void* k_pool, const void* v_pool,
                             const float* k_scale, const float* v_scale, int64_t num_blocks,
                             int block_size, int num_kv_heads, int head_dim) {
    return pool_create(out, k_pool, v_pool, k_scale, v_scale, 0, num_blocks, block_size,
                       num_kv_heads, head_dim, PGD_FP8_E4M3);
}

int paged_kv_pool_create_q8(pgd_pool_t* out, const void* k_pool, const void* v_pool, int code,
                            const float* k_scale, const float* v_scale, int granularity,
                            int64_t num_blocks, int block_size, int num_kv_heads, int head_dim) {
    if (out) *out = nullptr;
    if (!is_q8(code)) return PGD_ERR_DTYPE;
    if (granularity != PGD_SCALE_PER_HEAD && granularity != PGD_SCALE_PER_BLOCK)
        return PGD_ERR_ARG;
    return pool_create(out, k_pool, v_pool, k_scale, v_scale,
                       granularity == PGD_SCALE_PER_BLOCK ? 1 : 0, num_blocks, block_size,
                       num_kv_heads, head_dim, code);
}

int paged_kv_pool_destroy(pgd_pool_t pool) {
    if (!pool) return PGD_OK;
    int rc = PGD_OK;
    {
        DeviceGuard g(pool->p.device);
        if (!g.ok || cudaFree(pool->p.err) != cudaSuccess) rc = PGD_ERR_CUDA;
    }
    delete pool;
    return rc;
}

int paged_gqa_auto_splits(pgd_pool_t pool, int* num_splits) {
    if (!pool || !num_splits) return PGD_ERR_ARG;
    *num_splits = resolve_parts(pool->p, 0);
    return PGD_OK;
}

int paged_gqa_workspace_size_ex(pgd_pool_t pool, int B, int q_len, int Hq, int num_splits,
                                size_t* bytes) {
    if (!pool || !bytes || B < 0 || q_len < 1 || Hq < 1 || num_splits < 0 ||
        num_splits > (1 << 20))
        return PGD_ERR_ARG;
    const Pool& p = pool->p;
    if (Hq % p.hkv != 0) return PGD_ERR_SHAPE;
    const int rows = q_len * (Hq / p.hkv);
    if (rows > kMaxGroup) return PGD_ERR_SHAPE;
    *bytes = workspace_layout(B, p.hkv, rows, choose_hg(p, rows), p.d,
                              resolve_parts(p, num_splits)).total;
    return PGD_OK;
}

int paged_gqa_workspace_size(pgd_pool_t pool, int B, int Hq, int num_splits, size_t* bytes) {
    return paged_gqa_workspace_size_ex(pool, B, 1, Hq, num_splits, bytes);
}

namespace {
// The decode of paged_gqa_decode_ex; out_on_host: `out` is host memory written
// through its mapped address (paged_gqa_decode_host), where the merge stays
// fused in the decode kernel (a second kernel's writes would cross the host
// link after the first one's: measured slower end to end).
int decode_ex_impl(pgd_pool_t pool, const void* q, int B, int q_len, int Hq,
                   const int32_t* block_table, int max_blocks, const int32_t* seq_lens,
                   int window, float scale, void* out, void* workspace, size_t workspace_bytes,
                   int num_splits, void* stream, bool out_on_host) {
    if (!pool) return PGD_ERR_ARG;
    const Pool& p = pool->p;
    Plan plan;
    WorkspaceLayout wl;
    {
        const int rc = check_decode(p, q, B, q_len, Hq, block_table, max_blocks, seq_lens, window,
                                    scale, out, workspace, workspace_bytes, num_splits, &plan,
                                    &wl);
        if (rc != PGD_OK) return rc;
    }
    if (B == 0) return PGD_OK;
    if (out_on_host && plan.merge_variant == 2) plan.merge_variant = 0;
    const int G = Hq / p.hkv;
    const int parts = plan.parts;
    const int hg = plan.hg;

    DeviceGuard g(p.device);
    if (!g.ok) return PGD_ERR_CUDA;

    DecodeArgs a;
    memset(&a, 0, sizeof(a));
    a.q = q;
    a.k_pool = p.k;
    a.v_pool = p.v;
    a.out = out;
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.B = B;
    a.q_len = q_len;
    a.window = window;
    a.hq = Hq;
    a.hkv = p.hkv;
    a.group = G;
    a.d = p.d;
    a.block_size = p.block_size;
    a.max_blocks = max_blocks;
    a.num_blocks = p.num_blocks;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.k_scale = p.k_scale;
    a.v_scale = p.v_scale;
    a.scale_per_block = p.scale_per_block;
    a.num_parts = parts;
    a.auto_parts = num_splits == 0;
    a.hg = hg;
    a.units = p.hkv / hg;
    a.tile_tokens = plan.tile_tokens;
    a.run_cost = p.dtype == PGD_F32 ? 0 : kRunCostTiles;  // the float32 path's merge kernel: 0
    a.err = p.err;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    a.counters = reinterpret_cast<int*>(ws + wl.counters_off);
    a.merge_variant = plan.merge_variant == 3 ? 0 : plan.merge_variant;
    a.tile_base = reinterpret_cast<int64_t*>(ws + wl.tile_base_off);
    a.part_lse = reinterpret_cast<float*>(ws + wl.part_lse_off);
    a.part_o = reinterpret_cast<float*>(ws + wl.part_o_off);

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (p.dtype != PGD_F32) {
        // the TMA kernel merges split runs itself, except in the separate-merge
        // variant, whose partials a second kernel merges over all SMs
        if (launch_decode_tma(a, p, s) != cudaSuccess) return PGD_ERR_CUDA;
        if (a.merge_variant == 2 && launch_merge_runs(a, s) != cudaSuccess) return PGD_ERR_CUDA;
    } else {
        if (launch_decode_simple(a, p.dtype, s) != cudaSuccess) return PGD_ERR_CUDA;
        if (launch_merge(a, p.dtype, s) != cudaSuccess) return PGD_ERR_CUDA;
    }
    return PGD_OK;
}
}  // namespace

int paged_gqa_decode_ex(pgd_pool_t pool, const void* q, int B, int q_len, int Hq,
                        const int32_t* block_table, int max_blocks, const int32_t* seq_lens,
                        int window, float scale, void* out, void* workspace,
                        size_t workspace_bytes, int num_splits, void* stream) {
    return decode_ex_impl(pool, q, B, q_len, Hq, block_table, max_blocks, seq_lens, window, scale,
                          out, workspace, workspace_bytes, num_splits, stream, false);
}

int paged_gqa_decode(pgd_pool_t pool, const void* q, int B, int Hq, const int32_t* block_table,
                     int max_blocks, const int32_t* seq_lens, float scale, void* out,
                     void* workspace, size_t workspace_bytes, int num_splits, void* stream) {
    return paged_gqa_decode_ex(pool, q, B, 1, Hq, block_table, max_blocks, seq_lens, 0, scale,
                               out, workspace, workspace_bytes, num_splits, stream);
}

// Staging room for paged_gqa_decode_host, after the decode workspace.
struct HostLayout {
    size_t io_bytes;   // q or out
    size_t bt_bytes;   // block_table
    size_t q_off, bt_off, sl_off, out_off, total;
};

static HostLayout host_layout(const Pool& p, size_t decode_bytes, int B, int q_len, int Hq,
                              int max_blocks) {
    HostLayout h;
    const size_t elt = p.dtype == PGD_F32 ? 4 : 2;
    h.io_bytes = (size_t)B * q_len * Hq * p.d * elt;
    h.bt_bytes = (size_t)B * max_blocks * sizeof(int32_t);
    h.q_off = round_up(decode_bytes, 256);
    h.bt_off = h.q_off + round_up(h.io_bytes, 256);
    h.sl_off = h.bt_off + round_up(h.bt_bytes, 256);
    h.out_off = h.sl_off + round_up((size_t)B * sizeof(int32_t), 256);
    h.total = h.out_off + round_up(h.io_bytes, 256);
    return h;
}

// The address through which kernels on `dev` reach `h`, when `h` is
// page-locked host memory mapped into the device's address space (or memory
// of `dev` itself, or managed memory) and aligned to `align`; nullptr when it
// has to be staged (pageable host memory, another device's memory).
static const void* kernel_address(const void* h, uintptr_t align, int dev) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, h) != cudaSuccess) {
        cudaGetLastError();  // the failed query's error is not sticky: clear it
        return nullptr;
    }
    if (at.type == cudaMemoryTypeUnregistered || !at.devicePointer) return nullptr;
    if (at.type == cudaMemoryTypeDevice && at.device != dev) return nullptr;
    return aligned(at.devicePointer, align) ? at.devicePointer : nullptr;
}

int paged_gqa_workspace_size_host(pgd_pool_t pool, int B, int q_len, int Hq, int max_blocks,
                                  int num_splits, size_t* bytes) {
    if (!pool || !bytes || max_blocks < 0) return PGD_ERR_ARG;
    size_t dec = 0;
    const int rc = paged_gqa_workspace_size_ex(pool, B, q_len, Hq, num_splits, &dec);
    if (rc != PGD_OK) return rc;
    *bytes = host_layout(pool->p, dec, B, q_len, Hq, max_blocks).total;
    return PGD_OK;
}

int paged_gqa_decode_host(pgd_pool_t pool, const void* h_q, int B, int q_len, int Hq,
                          const int32_t* h_block_table, int max_blocks,
                          const int32_t* h_seq_lens, int window, float scale, void* h_out,
                          void* workspace, size_t workspace_bytes, int num_splits,
                          void* stream) {
    if (!pool || max_blocks < 0) return PGD_ERR_ARG;
    size_t dec = 0;
    int rc = paged_gqa_workspace_size_ex(pool, B, q_len, Hq, num_splits, &dec);
    if (rc != PGD_OK) return rc;
    if (B == 0)
        return paged_gqa_decode_ex(pool, h_q, B, q_len, Hq, h_block_table, max_blocks,
                                   h_seq_lens, window, scale, h_out, workspace, workspace_bytes,
                                   num_splits, stream);
    if (!h_q || !h_out || !h_block_table || !h_seq_lens || !workspace) return PGD_ERR_ARG;
    const Pool& p = pool->p;
    const HostLayout hl = host_layout(p, dec, B, q_len, Hq, max_blocks);
    if (!aligned(workspace, 256) || workspace_bytes < hl.total) return PGD_ERR_WORKSPACE;

    DeviceGuard g(p.device);
    if (!g.ok) return PGD_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    // Inputs: read in place through the mapped address, else copied in first.
    auto input = [&](const void* h, uintptr_t align, size_t off, size_t n) -> const void* {
        if (const void* d = kernel_address(h, align, p.device)) return d;
        if (n && cudaMemcpyAsync(ws + off, h, n, cudaMemcpyDefault, s) != cudaSuccess)
            return nullptr;
        return ws + off;
    };
    const void* q = input(h_q, 16, hl.q_off, hl.io_bytes);
    const void* bt = input(h_block_table, 4, hl.bt_off, hl.bt_bytes);
    const void* sl = input(h_seq_lens, 4, hl.sl_off, (size_t)B * sizeof(int32_t));
    if (!q || !bt || !sl) return PGD_ERR_CUDA;
    void* out = const_cast<void*>(kernel_address(h_out, 16, p.device));
    const bool copy_out = out == nullptr;
    if (copy_out) out = ws + hl.out_off;
    rc = decode_ex_impl(pool, q, B, q_len, Hq, static_cast<const int32_t*>(bt), max_blocks,
                        static_cast<const int32_t*>(sl), window, scale, out, workspace, dec,
                        num_splits, stream, !copy_out);
    if (rc != PGD_OK) return rc;
    if (copy_out && cudaMemcpyAsync(h_out, out, hl.io_bytes, cudaMemcpyDefault, s) != cudaSuccess)
        return PGD_ERR_CUDA;
    return PGD_OK;
}

int paged_gqa_plan(int dtype, int num_kv_heads, int head_dim, int num_sms, int B, int q_len,
                   int Hq, int num_splits, int window, int* plan) {
    if (!plan) return PGD_ERR_ARG;
    Plan pl;
    const int rc = make_plan(dtype, num_kv_heads, head_dim, num_sms, B, q_len, Hq, num_splits,
                             window, &pl);
    if (rc != PGD_OK) return rc;
    plan[0] = pl.hg;
    plan[1] = pl.m_tiles;
    plan[2] = pl.tile_tokens;
    plan[3] = pl.parts;
    plan[4] = pl.merge_variant;
    return PGD_OK;
}

int paged_gqa_get_error(pgd_pool_t pool, void* stream) {
    if (!pool) return PGD_ERR_ARG;
    DeviceGuard g(pool->p.device);
    if (!g.ok) return PGD_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int host = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) return PGD_ERR_CUDA;
    if (cudaMemcpy(&host, pool->p.err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return PGD_ERR_CUDA;
    if (host != 0 && cudaMemset(pool->p.err, 0, sizeof(int)) != cudaSuccess) return PGD_ERR_CUDA;
    return host;
}

const char* paged_gqa_strerror(int status) {
    switch (status) {
        case PGD_OK: return "ok";
        case PGD_ERR_ARG: return "invalid argument";
        case PGD_ERR_SHAPE: return "unsupported or inconsistent shape";
        case PGD_ERR_DTYPE: return "unsupported dtype";
        case PGD_ERR_ALIGN: return "pointer not aligned";
        case PGD_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case PGD_ERR_CUDA: return "CUDA call failed";
        case PGD_ERR_BLOCK_ID: return "block id out of range";
        case PGD_ERR_SEQ_LEN: return "sequence length out of range";
        case PGD_ERR_UNSUPPORTED: return "unsupported request";
        case PGD_ERR_TIMEOUT: return "device pipeline wait timed out";
        case PGD_ERR_TOO_LARGE:
            return "request needs more scratch than the fixed no-alloc scratch array holds";
        case PGD_ERR_NO_BLOCKS: return "no free block left in the pool";
        case PGD_ERR_NO_SEQ: return "unknown sequence id";
        case PGD_ERR_SEQ_EXISTS: return "sequence id already in use";
        case PGD_ERR_SEQ_FULL: return "sequence holds its maximum number of blocks";
        default: return "unknown status";
    }
}

}  // extern "C"
