// Device-side work partition shared by the decode kernels and the merge kernel.
//
// The KV work of one call is the sequence of T-token tiles of every
// (sequence b, unit u) pair, in the order b-major, then unit, then tile:
//
//     flat(b, u, i) = tile_base[b] + u * n_b + i,   n_b = ceil(L_b / T)
//
// A unit is a group of HG consecutive KV heads that one tile covers together
// (HG = 1 for the CUDA-core kernel, up to 8 for the TMA kernel, which reads a
// page slice for all heads of the group in one copy); a sequence has
// Hkv / HG units.
// CTA c of P takes the span [floor(c N / P), floor((c+1) N / P)) of the N
// tiles, so every CTA gets the same amount of KV bytes (to one tile) whatever
// the length mix.
//
// Run cost.  Starting a run inside a span costs that CTA time the tiles do
// not show (its query rows, the piece's epilogue, the arrival and usually the
// merge that follows): with run_cost = W > 0 each run is preceded by W
// virtual tiles that hold no work, and the spans are cut over this virtual
// sequence, so a span holding a run start gets W fewer real tiles.  A tile is
// then named by its virtual index:
//
//     vbase(b) = sum over b' < b of units * (n_b' + W)   (0 for n_b' = 0)
//     tile i of run (b, u) = vbase(b) + u * (n_b + W) + W + i
//
// and everything below (spans, piece owners, segment flags) works on virtual
// indices; W = 0 gives the plain tile sequence.  A (b, u) run that lies inside one span is finished by that
// CTA; a run cut by span boundaries leaves one partial result per piece, in
// slot 0 of a CTA (the piece that starts the CTA's span) or slot 1 (the piece
// that ends it), and a log-sum-exp merge combines them (inside the TMA kernel,
// after its tile loop; a separate merge kernel after the CUDA-core kernel).
// This is the split-KV scheme of FlashDecoding ("Modern LLM Inference ...",
// section 8.3 lists FlashDecoding kernels) with the splits placed by work
// rather than per sequence.
#pragma once

#include <stdint.h>

#include "pgd_internal.h"

namespace pgd {

__device__ __forceinline__ bool seq_len_ok(int L, int max_blocks, int block_size) {
    return L >= 0 && (int64_t)L <= (int64_t)max_blocks * block_size;
}

// First tile a sequence of length L needs: with q_len query tokens (the last
// q_len cached ones) and a window of the W most recent tokens per query, the
// earliest token read is max(0, L - q_len - W + 1); without a window, 0.
__device__ __forceinline__ int first_tile_of(int L, int T, int q_len, int window) {
    if (window <= 0) return 0;
    const int lo = L - q_len - window + 1;
    return lo > 0 ? lo / T : 0;
}

// Tiles of T tokens a sequence of length L walks (0 for L == 0 or a length out
// of range).
__device__ __forceinline__ int tiles_of(int L, int max_blocks, int block_size, int T, int q_len,
                                        int window) {
    if (!seq_len_ok(L, max_blocks, block_size) || L == 0) return 0;
    return (L + T - 1) / T - first_tile_of(L, T, q_len, window);
}

__device__ __forceinline__ int64_t span_begin(int64_t c, int64_t N, int64_t P) {
    return (c * N) / P;
}

// CTA whose span holds flat tile x (N > 0).  When P > N some spans are empty;
// the owners of consecutive tiles can then skip CTAs, which own nothing.
__device__ __forceinline__ int64_t span_owner(int64_t x, int64_t N, int64_t P) {
    return ((x + 1) * P - 1) / N;
}

__device__ __forceinline__ void latch_error(int* err, int code) {
    atomicCAS(err, 0, code);
}

// Virtual tiles of a sequence with n tiles per unit (see "Run cost" above).
__device__ __forceinline__ int64_t virtual_tiles(int n, int units, int run_cost) {
    return n > 0 ? (int64_t)units * (n + run_cost) : 0;
}

// Start of this CTA's span, found with a block-wide scan over the sequences.
struct SpanStart {
    int64_t n_total;   // N: virtual tiles of the call (the real ones when run_cost = 0)
    int64_t parts;     // spans in use (<= gridDim.x)
    int64_t r0, r1;    // this CTA's span (virtual indices)
    int b;             // sequence holding r0 (valid when r0 < r1)
    int64_t b_base;    // vbase(b): virtual index of the sequence's first slot
    int unit, i;       // run (b, unit) and its tile i: the first real tile at or after r0
    int n_tiles;       // real tiles of the span
    int run_cost;      // W in use (0 when the call has few tiles per span)
};

// A call charges run starts only when it has at least this many real tiles
// per span in use.
constexpr int kRunCostMinTiles = 8;

// Real tiles before virtual slot x + 1 counted from the start of sequence b
// (its runs are units of n tiles, each after W cost slots): tiles of the
// whole runs before x's run, plus those of x's run up to and including x.
__device__ __forceinline__ int real_upto(int64_t x, int64_t vbase, int n, int W) {
    const int off = (int)(x - vbase);
    const int per_run = n + W;
    const int i = off % per_run - W;  // tile of x in its run; < 0: a cost slot
    return (off / per_run) * n + (i < 0 ? 0 : i + 1);
}

// Every thread of the block must call this; blockDim.x is a multiple of 32 and
// at most 1024.  `scratch` is >= 96 int64 of shared memory, `out` a shared
// SpanStart.  With min_tiles > 1 the spans in use are min(parts,
// ceil(N / min_tiles)) (at least 1) and CTAs beyond them get an empty span;
// with min_tiles == 1 all `parts` spans are used (N counts real tiles there).
// The run cost asked for is used only when the call has at least
// kRunCostMinTiles real tiles per span in use (out->run_cost says which).
// CTA 0 also writes vbase[0..B] to global memory for the merge kernel.
__device__ inline void find_span_start(const int32_t* __restrict__ seq_lens, int B, int units,
                                       int T, int q_len, int window, int max_blocks,
                                       int block_size, int64_t parts, int min_tiles,
                                       int64_t* scratch, SpanStart* out,
                                       int64_t* __restrict__ tile_base_out, int run_cost = 0) {
    const int nt = blockDim.x;  // a multiple of 32
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5, nwarps = nt >> 5;
    const int per = (B + nt - 1) / nt;
    const int b_lo = min(B, tid * per);
    const int b_hi = min(B, b_lo + per);
    // tiles per unit of this thread's sequences (the first one kept: one
    // sequence per thread whenever B <= blockDim.x)
    const int n_first =
        b_lo < b_hi ? tiles_of(seq_lens[b_lo], max_blocks, block_size, T, q_len, window) : 0;
    auto tiles_at = [&](int b) {
        return b == b_lo ? n_first
                         : tiles_of(seq_lens[b], max_blocks, block_size, T, q_len, window);
    };
    // both prefixes in one scan: real tiles, and virtual tiles with the cost
    int64_t real_loc = 0, virt_loc = 0;
    for (int b = b_lo; b < b_hi; ++b) {
        const int n = tiles_at(b);
        real_loc += (int64_t)units * n;
        virt_loc += virtual_tiles(n, units, run_cost);
    }
    int64_t real_inc = real_loc, virt_inc = virt_loc;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int64_t r = __shfl_up_sync(0xffffffffu, real_inc, off);
        const int64_t v = __shfl_up_sync(0xffffffffu, virt_inc, off);
        if (lane >= off) {
            real_inc += r;
            virt_inc += v;
        }
    }
    if (lane == 31) {
        scratch[warp] = virt_inc;
        scratch[64 + warp] = real_inc;
    }
    __syncthreads();
    if (warp == 0) {
        int64_t v = lane < nwarps ? scratch[lane] : 0;
        int64_t r = lane < nwarps ? scratch[64 + lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int64_t v2 = __shfl_up_sync(0xffffffffu, v, off);
            const int64_t r2 = __shfl_up_sync(0xffffffffu, r, off);
            if (lane >= off) {
                v += v2;
                r += r2;
            }
        }
        if (lane < nwarps) {
            scratch[32 + lane] = v;   // inclusive prefixes of the warps
            scratch[64 + lane] = r;
        }
        if (lane == nwarps - 1) {
            const int64_t real = r;
            // spans in use, and the run cost: only where spans hold many tiles
            // (with a few tiles per span, cost slots would leave spans with none)
            int64_t p = parts;
            if (min_tiles > 1) {  // fewer spans only when asked for
                p = (real + min_tiles - 1) / min_tiles;
                p = p < parts ? p : parts;
                p = p > 0 ? p : 1;
            }
            const int W = real >= (int64_t)kRunCostMinTiles * p ? run_cost : 0;
            const int64_t n = W ? v : real;  // N
            out->n_total = n;
            out->run_cost = W;
            out->parts = p;
            out->r0 = blockIdx.x < p ? span_begin(blockIdx.x, n, p) : n;
            out->r1 = blockIdx.x < p ? span_begin(blockIdx.x + 1, n, p) : n;
            out->b = -1;
            out->b_base = 0;
            out->unit = out->i = 0;
            out->n_tiles = 0;
        }
    }
    __syncthreads();
    const int W = out->run_cost;
    const int64_t r0 = out->r0, r1 = out->r1;
    // this thread's exclusive prefixes, virtual (or real, without the cost)
    int64_t vrun = (warp ? (W ? scratch[32 + warp - 1] : scratch[64 + warp - 1]) : 0) +
                   (W ? virt_inc - virt_loc : real_inc - real_loc);
    int64_t rrun = (warp ? scratch[64 + warp - 1] : 0) + real_inc - real_loc;
    // real tiles before r0 and before r1, found by the threads whose
    // sequences hold those slots; their difference is the span's count
    for (int b = b_lo; b < b_hi; ++b) {
        const int nb = tiles_at(b);
        const int64_t n = virtual_tiles(nb, units, W);
        if (blockIdx.x == 0) tile_base_out[b] = vrun;
        if (r0 >= vrun && r0 < vrun + n) {
            const int off = (int)(r0 - vrun), per_run = nb + W;
            const int i = off % per_run - W;
            out->b = b;
            out->b_base = vrun;
            out->unit = off / per_run;
            out->i = i > 0 ? i : 0;
            scratch[96] = rrun + (off / per_run) * (int64_t)nb + (i > 0 ? i : 0);
        }
        if (r1 - 1 >= vrun && r1 - 1 < vrun + n && r0 < r1)
            scratch[97] = rrun + real_upto(r1 - 1, vrun, nb, W);
        vrun += n;
        rrun += (int64_t)units * nb;
    }
    if (blockIdx.x == 0 && tid == nt - 1) {
        tile_base_out[B] = out->n_total;    // then what a separate merge needs
        tile_base_out[B + 1] = out->parts;  // spans in use
        tile_base_out[B + 2] = out->run_cost;
    }
    __syncthreads();
    // (an empty span, r0 == r1, may still find a sequence holding r0: no count)
    if (tid == 0 && out->b >= 0 && r0 < r1) {
        const int64_t cnt = scratch[97] - scratch[96];
        out->n_tiles = cnt > 0 ? (int)cnt : 0;
    }
    __syncthreads();
}

// Cursor over the (b, unit, tile) sequence of one span.  Tile i of a run
// covers tokens [(first + i) T, (first + i + 1) T) of its sequence.
struct TileCursor {
    int b, unit, i, n_b;     // current position: tile i of n_b of (b, unit)
    int first;               // first tile of sequence b (windowed calls skip the start)
    int64_t run_start;       // virtual index of tile 0 of (b, unit); tile i is run_start + i
};

// Cursor at the first real tile at or after virtual index x, which sequence b
// (first slot b_base) holds; when x falls among a run's cost slots that is
// the run's tile 0.
__device__ inline TileCursor cursor_at_tile(int64_t x, int b, int64_t b_base,
                                            const int32_t* seq_lens, int T, int q_len,
                                            int window, int max_blocks, int block_size,
                                            int run_cost = 0) {
    TileCursor c;
    c.b = b;
    const int L = seq_lens[b];
    c.n_b = tiles_of(L, max_blocks, block_size, T, q_len, window);
    c.first = first_tile_of(L, T, q_len, window);
    const int per_run = c.n_b + run_cost;
    const int off = (int)(x - b_base);  // within one sequence: fits 32 bits
    c.unit = off / per_run;
    const int i = off % per_run - run_cost;
    c.i = i > 0 ? i : 0;
    c.run_start = b_base + (int64_t)c.unit * per_run + run_cost;
    return c;
}

// Cursor at the span's first real tile (the position find_span_start found).
__device__ inline TileCursor cursor_at(const SpanStart& s, const int32_t* seq_lens, int units,
                                       int T, int q_len, int window, int max_blocks,
                                       int block_size, int run_cost = 0) {
    (void)units;
    TileCursor c;
    c.b = s.b;
    const int L = seq_lens[s.b];
    c.n_b = tiles_of(L, max_blocks, block_size, T, q_len, window);
    c.first = first_tile_of(L, T, q_len, window);
    c.unit = s.unit;
    c.i = s.i;
    c.run_start = s.b_base + (int64_t)s.unit * (c.n_b + run_cost) + run_cost;
    return c;
}

// Next real tile: the next one of the run, else tile 0 of the next run (the
// next unit, or the first unit of the next sequence with tiles), which
// starts run_cost virtual slots after this run's end.
__device__ inline void cursor_next(TileCursor& c, const int32_t* seq_lens, int B, int units,
                                   int T, int q_len, int window, int max_blocks, int block_size,
                                   int run_cost = 0) {
    if (++c.i < c.n_b) return;
    c.run_start += c.n_b + run_cost;
    c.i = 0;
    if (++c.unit < units) return;
    c.unit = 0;
    int nb = 0;
    while (++c.b < B) {
        nb = tiles_of(seq_lens[c.b], max_blocks, block_size, T, q_len, window);
        if (nb > 0) break;
    }
    c.n_b = nb;
    if (c.b < B) c.first = first_tile_of(seq_lens[c.b], T, q_len, window);
}

// Segment flags for the piece of (b, unit) a CTA holds.
enum : int {
    kSegStart = 1,    // first tile of this CTA's piece of (b, unit)
    kSegEnd = 2,      // last tile of the piece
    kSegPartial = 4,  // piece is not the whole run: write a partial result
    kSegSlot1 = 8,    // partial goes to slot 1 (else slot 0)
    kTileBad = 16     // a block id of this tile was out of range
};

// Flags of tile x of run [run_start, run_start + n_b) inside span [r0, r1).
__device__ __forceinline__ int segment_flags(int64_t x, int64_t run_start, int n_b, int64_t r0,
                                             int64_t r1) {
    const int64_t run_end = run_start + n_b;
    const int64_t s0 = run_start > r0 ? run_start : r0;
    const int64_t s1 = run_end < r1 ? run_end : r1;
    int f = 0;
    if (x == s0) f |= kSegStart;
    if (x == s1 - 1) f |= kSegEnd;
    if (s0 != run_start || s1 != run_end) {
        f |= kSegPartial;
        if (s0 != r0) f |= kSegSlot1;
    }
    return f;
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float fast_log2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

}  // namespace pgd
