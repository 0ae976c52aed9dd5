// Internal declarations shared by the C-ABI layer (api.cpp) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "paged_gqa.h"

namespace pgd {

// Devices a process may use this library on (per-device state is kept in
// arrays of this size; pools on a device ordinal at or above it are refused).
constexpr int kMaxDevices = 64;

// Time a CTA spends on a run start that its tiles do not show (the piece's
// query rows, epilogue, arrival and, usually, a merge), in tiles of the TMA
// kernel (64 KB of K/V each): the work partition charges it to each run so
// that spans holding run starts get fewer tiles.  Measured by CTA timelines:
// a CTA with one more run start ended about three tiles later.
constexpr int kRunCostTiles = 3;

// Tokens per tile of the CUDA-core kernel (the TMA kernel uses 128 / HG).
constexpr int kSimpleTileTokens = 64;

// Largest query-head group the kernels handle (4 m16 row tiles).
constexpr int kMaxGroup = 64;
// A split run is merged by all its pieces' warps (shared merge, cooperative
// launch) only when one warp would need more than this many float4 loads per
// lane (six batches of 4 row passes x 4 pieces): below that, the waits and the
// second merge per CTA cost more than they save (measured).
constexpr int kShareMinLoads = 96;
// Separate merge (a second kernel after the decode) when each split run covers
// 2 to 5 spans, the runs times the head group fill the SMs and a head has at
// least this many query rows: then the merges fused at the end of the decode
// wait on pieces that end together, while the second kernel spreads them over
// every SM (measured; with longer runs the shared merge, with shorter ones or
// single rows the last arriver does better).
constexpr int kSepMinRows = 4;

struct Pool {
    const void* k;
    const void* v;
    int64_t num_blocks;
    int block_size;
    int hkv;
    int d;
    int dtype;
    int device;
    int num_sms;
    int* err;              // device error word (latched pgd_status)
    const float* k_scale;  // 8-bit pages: scales [Hkv] or [num_blocks][Hkv] (device), else null
    const float* v_scale;
    int scale_per_block;   // 8-bit pages: 1 when the scales are per block and KV head
    // bfloat16 TMA descriptors, one per head-group size HG = 1, 2, 4, 8 (index
    // log2 HG), valid where HG divides Hkv: 4-D view (d_lo 64, slot, head-half,
    // block) of the pool, box (64, min(bs, 128 / HG), HG * D / 64, 1).
    bool tmap_ok[4];
    CUtensorMap tmap_k[4];
    CUtensorMap tmap_v[4];
};

// Everything a decode launch needs, resolved on the host.
struct DecodeArgs {
    const void* q;
    const void* k_pool;
    const void* v_pool;
    void* out;
    const int32_t* block_table;
    const int32_t* seq_lens;
    int B;
    int q_len;             // query tokens per sequence (the last q_len cached tokens)
    int window;            // attend to the `window` most recent tokens per query; <= 0: all
    int hq;
    int hkv;
    int group;             // G = Hq / Hkv
    int d;
    int block_size;
    int max_blocks;
    int64_t num_blocks;
    float scale_log2;      // scale * log2(e): logits kept in base-2 units
    const float* k_scale;  // 8-bit pages: K / V scales per KV head [Hkv], or per physical
    const float* v_scale;  // block and KV head [num_blocks][Hkv] (device)
    int scale_per_block;   // which of the two
    int num_parts;         // CTAs of the decode grid (spans of the tile sequence)
    int auto_parts;        // num_parts came from num_splits == 0 (kernel may use fewer)
    int hg;                // KV heads per unit of work
    int units;             // units per sequence, Hkv / hg
    int tile_tokens;       // tokens per tile
    int run_cost;          // virtual tiles charged to each run start by the partition
    int* err;
    // workspace carve-up
    int* counters;         // [B][Hkv][m-tiles] per split run: pieces finished (zero between
                           // calls) and a flag bit flipped when the last piece arrives
    int merge_variant;     // host's choice of split-merge kernel variant: 0 last arriver,
                           // 1 shared (long runs; falls back to 0 when the grid cannot be
                           // resident), 2 separate run-merge kernel after the decode (many rows)
    int64_t* tile_base;    // [B + 3] first flat tile of each sequence, the total, the spans
                           // in use and the run cost
    float* part_o;         // [num_parts][2][hg * group][d] normalised partial outputs
    float* part_lse;       // [num_parts][2][hg * group]    partial log2-sum-exp
};

// The launch plan of a decode call, from shapes alone.
struct Plan {
    int hg;             // KV heads per unit of work
    int m_tiles;        // m16 row tiles of one head's query rows
    int tile_tokens;    // tokens per tile
    int parts;          // CTAs of the grid (spans of the tile sequence)
    int merge_variant;  // 0 last arriver, 1 shared (cooperative), 2 separate run merge,
                        // 3 float32 merge kernel
};

// Workspace layout for (B, G, D, parts); returns total bytes and fills offsets.
struct WorkspaceLayout {
    size_t counters_off, tile_base_off, part_lse_off, part_o_off, total;
};
// `rows` = query rows per KV head: q_len * G.
WorkspaceLayout workspace_layout(int B, int hkv, int rows, int hg, int d, int parts);

// Every argument check of a decode call (paged_gqa_decode_ex's contract), in
// the order the entry points apply them; fills the plan and, for B > 0, the
// workspace layout.  PGD_OK, or the status the call returns before anything
// is enqueued.
int check_decode(const Pool& p, const void* q, int B, int q_len, int Hq,
                 const int32_t* block_table, int max_blocks, const int32_t* seq_lens, int window,
                 float scale, const void* out, const void* workspace, size_t workspace_bytes,
                 int num_splits, Plan* plan, WorkspaceLayout* wl);

// KV heads per unit of work for this pool and rows per KV head.
int choose_hg(const Pool& p, int rows);

// The description behind a pool handle.
const Pool& pool_desc(pgd_pool_t h);

// Kernel launchers (return a cudaError_t from the launch).
cudaError_t launch_decode_simple(const DecodeArgs& a, int dtype, cudaStream_t s);
cudaError_t launch_decode_tma(const DecodeArgs& a, const Pool& p, cudaStream_t s);
cudaError_t launch_merge(const DecodeArgs& a, int dtype, cudaStream_t s);
cudaError_t launch_merge_runs(const DecodeArgs& a, cudaStream_t s);

}  // namespace pgd
