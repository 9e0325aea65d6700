// clo_attention.cu -- GQA decode attention for sm_103a over
//   (a) CLO's two KV sources, read in place: the top-k Cache Buffer (rows
//       picked by per-head token indices) and the full-length Persistent
//       Cache ("CLO: CPU-Light KVCache Offloading", section 2 hybrid attention
//       kernel; section 3 Fig. 9), and
//   (b) a paged block pool with a per-request block table (NEO's paged decode
//       attention; FastDecode's R-Part attention),
// computing softmax(q K^T / sqrt(d)) V per query head (KVPR page, section A3).
//
// Design (one GPU, HBM-bound):
//  * Work unit: a 16-token tile of one "segment" (one batch row / request and
//    one KV head).  The tiles form one stream per part (hybrid: the
//    contiguous Persistent Cache tiles, then the indexed Cache Buffer tiles;
//    paged: one part), and every part is cut into C equal contiguous ranges,
//    one per CTA (C = SMs x CTAs per SM, one wave).  Every CTA therefore
//    streams the same mix of contiguous and scattered bytes whether a tile
//    comes from a 128K-token persistent head or a 13K-row top-k head.  Odd
//    CTAs take their two ranges in the opposite order, so the grid never
//    switches from contiguous to scattered rows all at once.
//  * Three CTAs of four warps share an SM; the warps take their CTA's tiles
//    round-robin.  Each warp keeps a 2-stage shared-memory ring filled by
//    16-byte cp.async copies with an L2 evict-first hint (K and V rows of a
//    tile: 8 KB), one tile in flight while it computes the previous one.
//    Rows are XOR-swizzled in 16-byte chunks so ldmatrix reads are bank-
//    conflict free.  Indexed rows (Cache Buffer) and block-table rows cost the
//    same number of copies as contiguous rows: every copy is a whole
//    256-byte row.
//  * Math on the tensor cores with mma.sync m16n8k16 (fp16 in, fp32 accum):
//    S = K_tile Q^T puts the 16 tokens on M and the G <= 8 query heads of the
//    KV group on N (one n8 tile), then O^T += V_tile^T P^T puts the 128 head
//    dimensions on M and the heads on N.  P is moved from the S accumulator
//    layout to the B-operand layout with movmatrix.trans.  Online softmax in
//    the exp2 domain with per-tile warp-shuffle max.
//  * Each CTA merges its warps' (m, l, O) in shared memory whenever its range
//    crosses a segment end.  A segment that lies wholly in one CTA is written
//    straight to the output; a segment cut by CTA boundaries leaves one fp32
//    partial per CTA in the workspace (slot c + s + part * C, unique because
//    both partitions are contiguous) and a second small kernel merges those
//    partials by log-sum-exp.  That merge launch can also carry the next
//    layer's lookup (clo_hybrid_decode_attn_lookup).
//  * Every kernel uses programmatic dependent launch, so each grid becomes
//    resident while its predecessor drains.
//  * Bad indices, block-table entries, context lengths or persistent ids are
//    never dereferenced: the copy is zero-filled, the row masked, an error bit
//    is ORed into err_flag and the affected outputs are written as zeros.
#include <math.h>

#include <algorithm>
#include <mutex>

#include "clo_device.cuh"
#include "clo_fill.cuh"
#include "clo_lookup.cuh"

namespace clo {

constexpr int D = 128;
constexpr int TILE = 16;
constexpr int ROW_BYTES = D * 2;
constexpr int KV_TILE_BYTES = TILE * ROW_BYTES;  // 4 KB of K (or V) per tile
constexpr int STAGE_BYTES = 2 * KV_TILE_BYTES;   // K + V
constexpr int MAXG = 8;
constexpr int OSTRIDE = D + 4;  // padded merge-area row (floats): conflict-free writes
// Shape of the main kernel (overridable at build time): warps per CTA, ring
// stages per warp, CTAs per SM.  Shared memory per CTA is about
// warps * stages * 8 KB plus the merge area.
#ifndef CLO_ATTN_WARPS
#define CLO_ATTN_WARPS 4
#endif
#ifndef CLO_ATTN_STAGES
#define CLO_ATTN_STAGES 2
#endif
#ifndef CLO_ATTN_REVERSE_ODD
#define CLO_ATTN_REVERSE_ODD 1
#endif
#ifndef CLO_ATTN_CTAS_PER_SM
#define CLO_ATTN_CTAS_PER_SM 3
#endif
// Persistent Cache tiles a CTA that starts on the Cache Buffer brings into L2
// at its start (see attn_split_kernel).
#ifndef CLO_ATTN_EARLY_L2_TILES
#define CLO_ATTN_EARLY_L2_TILES 8
#endif
constexpr int ATTN_WARPS = CLO_ATTN_WARPS;
constexpr int ATTN_CTAS_PER_SM = CLO_ATTN_CTAS_PER_SM;
constexpr int ATTN_STAGES = CLO_ATTN_STAGES;
constexpr int ATTN_THREADS = ATTN_WARPS * 32;
constexpr int MERGE_THREADS = 512;
constexpr int MAX_HKV_HYBRID = 64;
constexpr int MAX_PAGED_B = 4096;
constexpr int MAX_ROWS = 1 << 24;  // rows per head: row offsets stay 32-bit
constexpr int SMEM_LIMIT = 227 * 1024;     // per CTA
constexpr int SMEM_PER_SM = 228 * 1024;    // per SM, 1 KB of it reserved per resident CTA
constexpr int MERGE_SMEM_LIMIT = 96 * 1024;

// One token set: batch row (or request) b, KV head kv.
struct Seg {
    int b;
    int kv;
    int slot;          // hybrid: persistent-cache slot, or -1 for the Cache Buffer
    int n_tok;         // tokens in the set
    int ntiles;        // ceil(n_tok / 16)
    long long first;   // index of its first tile in the flat stream
};

// Output side shared by both geometries.
struct AttnOut {
    const clo_half* q;
    clo_half* out;
    float* lse;
    float* ws_o;    // [slots][G][D] fp32 normalised partial outputs
    float* ws_lse;  // [slots][G] fp32 partial log2-sum-exp (+inf marks bad data)
    int32_t* err_flag;
    float scale_log2;
    int Hq;
    int G;
};

// ---------------------------------------------------------------- hybrid geometry
// The tile stream has two parts, each cut evenly over all CTAs: part 0 holds
// every Persistent Cache segment (ordered b, slot; T contiguous rows each),
// part 1 every Cache Buffer segment (ordered b, slot; k indexed rows each).
// Each CTA thus streams the same share of contiguous and of scattered rows,
// so no SM is left with only the slower scattered reads.  Slots [0, Np) are
// the persistent heads in persist_ids order, slots [Np, Hkv) the remaining
// KV heads in ascending order.
struct HybridGeo {
    const clo_half* cbK;
    const clo_half* cbV;
    const int32_t* idx;
    const clo_half* pK;
    const clo_half* pV;
    const int32_t* persist_ids;
    int k, C, Np, T, B, Hkv;
    int tp, tc;             // tiles of a persistent / Cache Buffer segment
    long long n0;           // tiles in part 0 (B * Np * tp)
    long long n1;           // tiles in part 1 (B * (Hkv - Np) * tc)

    static constexpr int kParts = 2;
    static constexpr bool kAheadAtFlush = false;
    // Shared scratch: [0] = ids valid flag, [1 .. Hkv] slot -> KV head,
    // [1 + Hkv .. 1 + 2 Hkv) staged persist_ids.
    static size_t smem_ints(int Hkv_, int /*B*/) { return 2 * static_cast<size_t>(Hkv_) + 4; }

    // This thread's share of persist_ids (thread j < Np loads entry j); issued
    // ahead of the bulk copies so it does not queue behind them.
    __device__ int ids_preload() const {
        return static_cast<int>(threadIdx.x) < Np ? __ldg(persist_ids + threadIdx.x) : 0;
    }
    __device__ void cta_init(int* sm, int32_t* err_flag, bool report) const {
        cta_init_with(sm, err_flag, report, ids_preload());
    }
    __device__ void cta_init_with(int* sm, int32_t* err_flag, bool report, int id) const {
        // sm[1 + Hkv + j] stages persist_ids so thread 0 does not wait on Np loads in turn.
        if (static_cast<int>(threadIdx.x) < Np) sm[1 + Hkv + threadIdx.x] = id;
        __syncthreads();
        if (threadIdx.x == 0) {
            unsigned long long used = 0ull;
            int ok = 1;
            for (int j = 0; j < Np; ++j) {
                const int g = sm[1 + Hkv + j];
                if (g < 0 || g >= Hkv || ((used >> g) & 1ull)) {
                    ok = 0;
                    sm[1 + j] = 0;
                } else {
                    used |= 1ull << g;
                    sm[1 + j] = g;
                }
            }
            int slot = Np;
            for (int g = 0; g < Hkv && slot < Hkv; ++g)
                if (!((used >> g) & 1ull)) sm[1 + slot++] = g;
            if (!ok)  // keep a permutation so every output row is still written (as zeros)
                for (int j = 0; j < Hkv; ++j) sm[1 + j] = j;
            sm[0] = ok;
            if (!ok && report) report_error(err_flag, CLO_FLAG_BAD_PERSIST);
        }
    }
    // Segment boundaries do not depend on device data.
    static constexpr bool kStaticLayout = true;
    __device__ long long part_begin(int p, const int*) const { return p == 0 ? 0 : n0; }
    __device__ long long part_tiles(int p, const int*) const { return p == 0 ? n0 : n1; }
    __device__ long long num_tiles(const int*) const { return n0 + n1; }
    __device__ int seg_of(long long t, const int*) const {
        if (t < n0) {
            const long long per_b = static_cast<long long>(Np) * tp;
            const int b = static_cast<int>(t / per_b);
            const int slot = static_cast<int>((t - per_b * b) / tp);
            return b * Np + slot;
        }
        const long long t1 = t - n0;
        const int nc = Hkv - Np;
        const long long per_b = static_cast<long long>(nc) * tc;
        const int b = static_cast<int>(t1 / per_b);
        const int j = static_cast<int>((t1 - per_b * b) / tc);
        return B * Np + b * nc + j;
    }
    __device__ long long segment_first(int s) const {
        return s < B * Np ? static_cast<long long>(s) * tp
                          : n0 + static_cast<long long>(s - B * Np) * tc;
    }
    __device__ int segment_part(int s) const { return s < B * Np ? 0 : 1; }
    // KV head of token set s from persist_ids, computed by one warp without
    // a shared table: lane j holds entries j and j + 32 (-1 past Np, loaded
    // with ids_warp_load).  ids_ok = the ids are distinct and in range (else
    // the slots map to heads 0..Hkv-1 in order, as in cta_init).
    __device__ void ids_warp_load(int lane, int& id0, int& id1) const {
        id0 = lane < Np ? __ldg(persist_ids + lane) : -1;
        id1 = lane + 32 < Np ? __ldg(persist_ids + lane + 32) : -1;
    }
    __device__ int segment_kv_warp(int s, int lane, int id0, int id1, bool& ids_ok) const {
        const bool in0 = lane < Np, in1 = lane + 32 < Np;
        const bool bad = (in0 && (id0 < 0 || id0 >= Hkv)) || (in1 && (id1 < 0 || id1 >= Hkv));
        unsigned long long mine = 0ull;
        if (in0 && !bad) mine |= 1ull << id0;
        if (in1 && !bad) mine |= 1ull << id1;
        const unsigned lo = __reduce_or_sync(FULL_MASK, static_cast<unsigned>(mine));
        const unsigned hi = __reduce_or_sync(FULL_MASK, static_cast<unsigned>(mine >> 32));
        const unsigned long long used = (static_cast<unsigned long long>(hi) << 32) | lo;
        ids_ok = !__any_sync(FULL_MASK, bad) && __popcll(used) == Np;  // no duplicates
        const int slot = s < B * Np ? s % Np : Np + (s - B * Np) % (Hkv - Np);
        const int own = __shfl_sync(FULL_MASK, slot < 32 ? id0 : id1, slot & 31);
        if (!ids_ok) return slot;
        if (slot < Np) return own;
        int left = slot - Np;
        for (int g = 0; g < Hkv; ++g)
            if (!((used >> g) & 1ull) && left-- == 0) return g;
        return 0;
    }
    // Upper bound on the CTA ranges one token set can span (host side).
    long long max_partials_host(int C) const {
        long long most = 1;
        if (n0 > 0) most = std::max(most, (static_cast<long long>(tp) * C + n0 - 1) / n0 + 1);
        if (n1 > 0) most = std::max(most, (static_cast<long long>(tc) * C + n1 - 1) / n1 + 1);
        return most;
    }
    __device__ int segment_ntiles(int s) const { return s < B * Np ? tp : tc; }
    __host__ __device__ int num_segments() const { return B * Hkv; }
    __device__ Seg segment(int s, const int* sm, bool no_kv = false) const {
        Seg g;
        int slot;
        if (s < B * Np) {
            g.b = s / Np;
            slot = s - g.b * Np;
            g.n_tok = T;
            g.ntiles = tp;
            g.first = static_cast<long long>(s) * tp;
            g.slot = slot;
        } else {
            const int nc = Hkv - Np;
            const int s1 = s - B * Np;
            g.b = s1 / nc;
            const int j = s1 - g.b * nc;
            slot = Np + j;
            g.n_tok = k;
            g.ntiles = tc;
            g.first = n0 + static_cast<long long>(s1) * tc;
            g.slot = -1;
        }
        g.kv = no_kv ? 0 : sm[1 + slot];
        return g;
    }
    __device__ bool all_bad(const int* sm) const { return sm[0] == 0; }
    // Brings the K and V rows of Persistent Cache tiles [t0, t0 + n) (part 0)
    // into L2 with an evict-last hint; needs no device data.
    __device__ void prefetch_persistent(long long t0, long long n) const {
        constexpr int kLines = KV_TILE_BYTES / 128;  // 128-byte lines of K (or V) in a tile
        for (long long i = threadIdx.x; i < n * 2 * kLines; i += blockDim.x) {
            const long long t = t0 + i / (2 * kLines);
            const int line = static_cast<int>(i % (2 * kLines));
            const int s = static_cast<int>(t / tp);
            const int tile_in = static_cast<int>(t - static_cast<long long>(s) * tp);
            const int row = tile_in * TILE + (line % kLines) / 2;  // two lines a 256-byte row
            if (row >= T) continue;
            const clo_half* base = (line < kLines ? pK : pV) + static_cast<long long>(s) * T * D;
            prefetch_l2_keep(base + static_cast<long long>(row) * D + (line & 1) * 64);
        }
    }
    // Brings the Cache Buffer indices of tiles [t0, t0 + n) of part 1 into L2
    // (the lines holding each tile's first and last index), so that the
    // per-tile index loads, issued one pipeline step ahead of their copies,
    // hit L2 instead of waiting on DRAM behind the K/V stream.  Needs the slot
    // table (cta_init).
    __device__ void prefetch_indices(const int* sm, long long t0, long long n) const {
        for (long long i = threadIdx.x; i < n; i += blockDim.x) {
            const Seg g = segment(seg_of(t0 + i, sm), sm);
            const int tok = static_cast<int>(t0 + i - g.first) * TILE;
            const int32_t* row = idx + (static_cast<long long>(g.b) * Hkv + g.kv) * k;
            prefetch_l2(row + tok);
            prefetch_l2(row + min(tok + TILE - 1, k - 1));
        }
    }
    // The indirection of row r (0..15) of a tile: its Cache Buffer index
    // (0 for persistent rows and rows past the end).  Issued one pipeline
    // step before the row is copied so its latency overlaps the math.
    __device__ int row_load(const Seg& g, int tile_in, int r) const {
        const int tok = tile_in * TILE + r;
        if (g.slot >= 0 || tok >= g.n_tok) return 0;
        return __ldg(idx + (static_cast<long long>(g.b) * Hkv + g.kv) * k + tok);
    }
    // Row r of tile `tile_in` of segment g: the segment's K/V base (uniform over
    // the tile) and the row's element offset from it (< 2^31: C, T <= 2^24);
    // in_range = the token exists, ok = its address is valid.
    __device__ void row(const Seg& g, int tile_in, int r, int raw, const int* sm,
                        const clo_half*& bk, const clo_half*& bv, int& roff, bool& in_range,
                        bool& ok) const {
        const int tok = tile_in * TILE + r;
        in_range = tok < g.n_tok;
        if (g.slot >= 0) {
            const long long base = (static_cast<long long>(g.b) * Np + g.slot) * T * D;
            bk = pK + base;
            bv = pV + base;
            roff = tok * D;
            ok = true;  // slot-addressed: valid even if persist_ids is not (outputs zeroed then)
        } else {
            const long long base = (static_cast<long long>(g.b) * Hkv + g.kv) * C * D;
            bk = cbK + base;
            bv = cbV + base;
            ok = (sm[0] != 0) && raw >= 0 && raw < C;
            roff = (ok ? raw : 0) * D;
        }
    }
};

// ---------------------------------------------------------------- paged geometry
// Segments are ordered (request r, KV head h), each ceil(ctx_len[r]/16) tiles.
struct PagedGeo {
    const clo_half* kc;
    const clo_half* vc;
    const int32_t* block_table;
    const int32_t* ctx_len;
    int max_blocks, num_blocks, B, Hkv;

    // Shared scratch: prefix[0 .. B] (tiles before request r, all heads) and
    // 32 ints for the block scan.
    static size_t smem_ints(int /*Hkv*/, int B_) { return static_cast<size_t>(B_) + 1 + 40; }

    __device__ int tiles_of(int r) const {
        const int n = ctx_len[r];
        if (n < 0 || n > max_blocks * TILE) return -1;
        return (n + TILE - 1) / TILE;
    }

    __device__ void cta_init(int* sm, int32_t* err_flag, bool report) const {
        // Block-wide exclusive scan of Hkv * tiles(r) over r < B.
        int* prefix = sm;
        int* wsum = sm + B + 1;
        const int nt = blockDim.x;
        const int per = (B + nt - 1) / nt;
        const int r0 = threadIdx.x * per;
        const int r1 = min(B, r0 + per);
        int local = 0;
        bool bad = false;
        for (int r = r0; r < r1; ++r) {
            const int t = tiles_of(r);
            bad |= t < 0;
            local += (t < 0 ? 0 : t) * Hkv;
        }
        if (bad && report) report_error(err_flag, CLO_FLAG_BAD_CTX);
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        int incl = local;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(FULL_MASK, incl, off);
            if (lane >= off) incl += v;
        }
        if (lane == 31) wsum[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int nw = (nt + 31) / 32;
            int v = lane < nw ? wsum[lane] : 0;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int u = __shfl_up_sync(FULL_MASK, v, off);
                if (lane >= off) v += u;
            }
            if (lane < nw) wsum[lane] = v;  // inclusive over warps
        }
        __syncthreads();
        int run = (warp > 0 ? wsum[warp - 1] : 0) + incl - local;
        if (threadIdx.x == 0) prefix[0] = 0;
        for (int r = r0; r < r1; ++r) {
            const int t = tiles_of(r);
            run += (t < 0 ? 0 : t) * Hkv;
            prefix[r + 1] = run;
        }
    }
    static constexpr int kParts = 1;
    static constexpr bool kAheadAtFlush = true;
    static constexpr bool kStaticLayout = false;  // depends on ctx_len
    __device__ long long part_begin(int, const int*) const { return 0; }
    __device__ long long part_tiles(int, const int* sm) const { return sm[B]; }
    __device__ long long num_tiles(const int* sm) const { return sm[B]; }
    // Request owning tile t: the last r with prefix[r] <= t (skips empty requests).
    __device__ int request_of(long long t, const int* sm) const {
        int lo = 0, hi = B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (sm[mid] <= t) lo = mid; else hi = mid - 1;
        }
        return lo;
    }
    __device__ int seg_of(long long t, const int* sm) const {
        const int r = request_of(t, sm);
        const int tr = (sm[r + 1] - sm[r]) / Hkv;
        return r * Hkv + static_cast<int>((t - sm[r]) / tr);
    }
    __device__ long long segment_first(int) const { return 0; }  // unused: layout is dynamic
    __device__ int segment_part(int) const { return 0; }
    // Lengths live on the device: assume the worst case (one head per block).
    long long max_partials_host(int C) const { return static_cast<long long>(C); }
    __device__ int segment_ntiles(int) const { return 0; }
    __host__ __device__ int num_segments() const { return B * Hkv; }
    __device__ Seg segment(int s, const int* sm, bool = false) const {
        Seg g;
        g.b = s / Hkv;
        g.kv = s - g.b * Hkv;
        g.slot = -1;
        const int tr = (sm[g.b + 1] - sm[g.b]) / Hkv;
        g.ntiles = tr;
        g.n_tok = tr > 0 ? ctx_len[g.b] : 0;
        g.first = sm[g.b] + static_cast<long long>(g.kv) * tr;
        return g;
    }
    __device__ bool all_bad(const int*) const { return false; }
    __device__ void prefetch_indices(const int*, long long, long long) const {}
    // The block holding tile `tile_in` (the same for all 16 rows).
    __device__ int row_load(const Seg& g, int tile_in, int /*r*/) const {
        return __ldg(block_table + static_cast<long long>(g.b) * max_blocks + tile_in);
    }
    __device__ void row(const Seg& g, int tile_in, int r, int blk, const int*,
                        const clo_half*& bk, const clo_half*& bv, int& roff, bool& in_range,
                        bool& ok) const {
        ok = blk >= 0 && blk < num_blocks;
        const long long base = (static_cast<long long>(ok ? blk : 0) * Hkv + g.kv) * TILE * D;
        bk = kc + base;
        bv = vc + base;
        in_range = tile_in * TILE + r < g.n_tok;
        roff = r * D;
    }
};

// ---------------------------------------------------------------- tile copy
// Producer-side position in the segment order.  A warp's tiles increase, so
// the segment of the next tile is found by stepping forward from the last one
// (no per-tile division).
struct Cursor {
    int s;
    Seg sg;
};

template <class Geo>
__device__ __forceinline__ void cursor_init(const Geo& geo, const int* gsm, long long t, Cursor& c) {
    c.s = geo.seg_of(t, gsm);
    c.sg = geo.segment(c.s, gsm);
}

template <class Geo>
__device__ __forceinline__ void cursor_seek(const Geo& geo, const int* gsm, long long t, Cursor& c) {
    while (t >= c.sg.first + c.sg.ntiles) c.sg = geo.segment(++c.s, gsm);
}

// A tile whose segment is located and whose row indirection load is in
// flight; the copies are issued one pipeline step later.
struct Pending {
    Seg sg;
    int tile_in;
    int raw;
};

template <class Geo>
__device__ __forceinline__ void prefetch_tile(const Geo& geo, const int* gsm, long long t, int lane,
                                              Cursor& cur, Pending& pd) {
    cursor_seek(geo, gsm, t, cur);
    pd.sg = cur.sg;
    pd.tile_in = static_cast<int>(t - cur.sg.first);
    pd.raw = geo.row_load(pd.sg, pd.tile_in, lane & 15);
}

// Issues the cp.async copies of one tile (16 K rows + 16 V rows) into a ring
// stage and records its row masks (bits 0-15 valid rows, 16-31 bad rows).
// dry: every copy is a zero-fill that reads no global memory.
template <class Geo>
__device__ __forceinline__ void issue_tile(const Geo& geo, const int* gsm, const Pending& pd,
                                           uint32_t stage, uint32_t* mask_slot, int lane,
                                           uint64_t policy, bool dry = false) {
    const clo_half* bk;
    const clo_half* bv;
    int roff;
    bool in_range, ok;
    geo.row(pd.sg, pd.tile_in, lane & 15, pd.raw, gsm, bk, bv, roff, in_range, ok);
    const unsigned valid = __ballot_sync(FULL_MASK, in_range && ok) & 0xffffu;
    const unsigned bad = __ballot_sync(FULL_MASK, in_range && !ok) & 0xffffu;
    if (lane == 0) *mask_slot = valid | (bad << 16);
    const int chunk = lane & 15;
    const uint32_t dst0 = stage + (lane >> 4) * ROW_BYTES;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = (lane >> 4) + 2 * i;
        const int ro = __shfl_sync(FULL_MASK, roff, r) + chunk * 8;
        const bool v = (valid >> r) & 1u;
        const uint32_t dst = dst0 + 2 * i * ROW_BYTES + ((chunk ^ (r & 7)) << 4);
        const int nb = (v && !dry) ? 16 : 0;  // dry: zero-fill, nothing read
        cp_async_16_hint(dst, bk + (v ? ro : 0), nb, policy);
        cp_async_16_hint(dst + KV_TILE_BYTES, bv + (v ? ro : 0), nb, policy);
    }
}

// ---------------------------------------------------------------- tile math
struct WarpState {
    float m0, m1;      // running max (log2 domain) of heads 2c, 2c+1 (c = lane % 4)
    float l0, l1;      // this lane's partial softmax denominators
    float acc[8][4];   // O^T fragments: d rows 16i + lane/4 (+8), heads 2c, 2c+1
    int bad;
};

__device__ __forceinline__ void state_reset(WarpState& w) {
    w.m0 = w.m1 = -INFINITY;
    w.l0 = w.l1 = 0.f;
    w.bad = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) w.acc[i][j] = 0.f;
}

__device__ __forceinline__ void compute_tile(uint32_t st, uint32_t valid,
                                             const uint32_t (&qb)[8][2], float sl2,
                                             WarpState& w, int lane) {
    const uint32_t Ks = st, Vs = st + KV_TILE_BYTES;
    // Two accumulators over alternating k-steps halve the mma dependency chain.
    float s[4] = {0.f, 0.f, 0.f, 0.f}, s2[4] = {0.f, 0.f, 0.f, 0.f};
    const int arow = lane & 15;
    const int ahi = lane >> 4;
#pragma unroll
    for (int kk = 0; kk < 8; kk += 2) {
        uint32_t a[4], a2[4];
        const int chunk = 2 * kk + ahi;
        ldmatrix_x4(a, Ks + arow * ROW_BYTES + ((chunk ^ (arow & 7)) << 4));
        ldmatrix_x4(a2, Ks + arow * ROW_BYTES + (((chunk + 2) ^ (arow & 7)) << 4));
        mma_16816(s, a, qb[kk][0], qb[kk][1]);
        mma_16816(s2, a2, qb[kk + 1][0], qb[kk + 1][1]);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) s[j] += s2[j];
    const int r0 = lane >> 2;
    const bool v0 = (valid >> r0) & 1u;
    const bool v1 = (valid >> (r0 + 8)) & 1u;
    const float x0 = v0 ? s[0] * sl2 : -INFINITY;  // token r0,   head 2c
    const float x1 = v0 ? s[1] * sl2 : -INFINITY;  // token r0,   head 2c+1
    const float x2 = v1 ? s[2] * sl2 : -INFINITY;  // token r0+8, head 2c
    const float x3 = v1 ? s[3] * sl2 : -INFINITY;  // token r0+8, head 2c+1
    float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
    for (int off = 4; off <= 16; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(FULL_MASK, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(FULL_MASK, mx1, off));
    }
    const float mn0 = fmaxf(w.m0, mx0), mn1 = fmaxf(w.m1, mx1);
    const float ref0 = mn0 == -INFINITY ? 0.f : mn0;
    const float ref1 = mn1 == -INFINITY ? 0.f : mn1;
    const float al0 = fast_exp2(w.m0 - ref0), al1 = fast_exp2(w.m1 - ref1);
    const float p0 = fast_exp2(x0 - ref0), p2 = fast_exp2(x2 - ref0);
    const float p1 = fast_exp2(x1 - ref1), p3 = fast_exp2(x3 - ref1);
    w.l0 = fmaf(w.l0, al0, p0 + p2);
    w.l1 = fmaf(w.l1, al1, p1 + p3);
    w.m0 = mn0;
    w.m1 = mn1;
    if (__any_sync(FULL_MASK, al0 != 1.f || al1 != 1.f)) {  // the running max moved
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            w.acc[i][0] *= al0;
            w.acc[i][1] *= al1;
            w.acc[i][2] *= al0;
            w.acc[i][3] *= al1;
        }
    }
    const uint32_t pb0 = movmatrix_trans(pack_half2(p0, p1));  // tokens 0-7
    const uint32_t pb1 = movmatrix_trans(pack_half2(p2, p3));  // tokens 8-15
    const int vtok = (lane & 7) + ((lane >> 4) << 3);
    const int vsel = (lane >> 3) & 1;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t a[4];
        const int chunk = 2 * i + vsel;
        ldmatrix_x4_trans(a, Vs + vtok * ROW_BYTES + ((chunk ^ (vtok & 7)) << 4));
        mma_16816(w.acc[i], a, pb0, pb1);
    }
}

__device__ __forceinline__ void load_q(const AttnOut& o, const Seg& sg, int lane,
                                       uint32_t (&qb)[8][2]) {
    const int h = lane >> 2;
    const bool has = h < o.G;
    const clo_half* qrow =
        o.q + (static_cast<size_t>(sg.b) * o.Hq + static_cast<size_t>(sg.kv) * o.G + (has ? h : 0)) * D +
        2 * (lane & 3);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        qb[kk][0] = has ? __ldg(reinterpret_cast<const unsigned int*>(qrow + 16 * kk)) : 0u;
        qb[kk][1] = has ? __ldg(reinterpret_cast<const unsigned int*>(qrow + 16 * kk + 8)) : 0u;
    }
}

struct MergeSmem {
    float* m;     // [MAXG][WARPS]
    float* l;     // [MAXG][WARPS]
    int* bad;     // [WARPS]
    float* o;     // [WARPS][G][OSTRIDE]
};

// Combines the warps' states for segment s; writes the final output when the
// whole segment is inside this CTA, else this CTA's partial.
__device__ __forceinline__ void flush_segment(const AttnOut& o, const MergeSmem& ms, WarpState& w,
                                              const Seg& sg, int s, long long c0, long long c1,
                                              size_t slot_base, bool force_bad, int warp,
                                              int lane) {
    float l0 = w.l0, l1 = w.l1;
#pragma unroll
    for (int off = 4; off <= 16; off <<= 1) {
        l0 += __shfl_xor_sync(FULL_MASK, l0, off);
        l1 += __shfl_xor_sync(FULL_MASK, l1, off);
    }
    const int h0 = 2 * (lane & 3), h1 = h0 + 1;
    if (lane < 4) {  // [head][warp] layout: one 16-byte load per head in the merge below
        ms.m[h0 * ATTN_WARPS + warp] = w.m0;
        ms.m[h1 * ATTN_WARPS + warp] = w.m1;
        ms.l[h0 * ATTN_WARPS + warp] = l0;
        ms.l[h1 * ATTN_WARPS + warp] = l1;
    }
    const int badw = static_cast<int>(__reduce_or_sync(FULL_MASK, static_cast<unsigned>(w.bad)));
    if (lane == 0) {
        ms.bad[warp] = badw;
        if (badw != 0) report_error(o.err_flag, CLO_FLAG_BAD_INDEX);
    }
    const int G = o.G;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int d0 = 16 * i + (lane >> 2);
        if (h0 < G) {
            ms.o[(warp * G + h0) * OSTRIDE + d0] = w.acc[i][0];
            ms.o[(warp * G + h0) * OSTRIDE + d0 + 8] = w.acc[i][2];
        }
        if (h1 < G) {
            ms.o[(warp * G + h1) * OSTRIDE + d0] = w.acc[i][1];
            ms.o[(warp * G + h1) * OSTRIDE + d0 + 8] = w.acc[i][3];
        }
    }
    __syncthreads();
    // Each thread combines four consecutive columns of one head with 16-byte
    // shared loads: few load instructions matter here, because the other
    // CTAs' copies keep the SM's memory pipeline busy and every shared load
    // queues behind them.
    static_assert(ATTN_WARPS == 4, "the merge reads the warps' (m, l) of a head as one float4");
    const int4 bw = *reinterpret_cast<const int4*>(ms.bad);
    const bool bad = force_bad || (bw.x | bw.y | bw.z | bw.w) != 0;
    const bool complete = sg.first >= c0 && sg.first + sg.ntiles <= c1;
    for (int it = threadIdx.x; it < G * (D / 4); it += ATTN_THREADS) {
        const int h = it / (D / 4), dd = (it % (D / 4)) * 4;
        const float4 mv = *reinterpret_cast<const float4*>(ms.m + h * ATTN_WARPS);
        const float4 lv = *reinterpret_cast<const float4*>(ms.l + h * ATTN_WARPS);
        const float mx[4] = {mv.x, mv.y, mv.z, mv.w};
        const float lx[4] = {lv.x, lv.y, lv.z, lv.w};
        float4 ov[ATTN_WARPS];
#pragma unroll
        for (int x = 0; x < ATTN_WARPS; ++x)
            ov[x] = *reinterpret_cast<const float4*>(ms.o + (x * G + h) * OSTRIDE + dd);
        const float M = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
        float L = 0.f, O[4] = {0.f, 0.f, 0.f, 0.f};
        if (M != -INFINITY) {
#pragma unroll
            for (int x = 0; x < ATTN_WARPS; ++x) {
                if (mx[x] != -INFINITY) {
                    const float e = fast_exp2(mx[x] - M);
                    L = fmaf(lx[x], e, L);
                    O[0] = fmaf(ov[x].x, e, O[0]);
                    O[1] = fmaf(ov[x].y, e, O[1]);
                    O[2] = fmaf(ov[x].z, e, O[2]);
                    O[3] = fmaf(ov[x].w, e, O[3]);
                }
            }
        }
        const bool empty = !(L > 0.f);
        if (complete) {
            const size_t row = static_cast<size_t>(sg.b) * o.Hq + static_cast<size_t>(sg.kv) * G + h;
            uint32_t pk[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const float v0 = (bad || empty) ? 0.f : O[2 * j] / L;
                const float v1 = (bad || empty) ? 0.f : O[2 * j + 1] / L;
                pk[j] = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(v0))) |
                        (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(v1))) << 16);
            }
            *reinterpret_cast<uint2*>(o.out + row * D + dd) = make_uint2(pk[0], pk[1]);
            if (o.lse != nullptr && dd == 0)
                o.lse[row] = (bad || empty) ? -INFINITY : (M + log2f(L)) * LN2;
        } else {
            const size_t slot = slot_base + static_cast<size_t>(s);
            const float4 r = empty ? make_float4(0.f, 0.f, 0.f, 0.f)
                                   : make_float4(O[0] / L, O[1] / L, O[2] / L, O[3] / L);
            *reinterpret_cast<float4*>(o.ws_o + (slot * G + h) * D + dd) = r;
            if (dd == 0) o.ws_lse[slot * G + h] = bad ? INFINITY : (empty ? -INFINITY : M + log2f(L));
        }
    }
    __syncthreads();
}

template <class Geo>
__global__ void __launch_bounds__(ATTN_THREADS, ATTN_CTAS_PER_SM)
    attn_split_kernel(const Geo geo, const AttnOut o) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int RING = ATTN_WARPS * ATTN_STAGES * STAGE_BYTES;
    uint32_t* masks = reinterpret_cast<uint32_t*>(smem + RING);
    MergeSmem ms;
    ms.m = reinterpret_cast<float*>(masks + ATTN_WARPS * ATTN_STAGES);
    ms.l = ms.m + ATTN_WARPS * MAXG;
    ms.bad = reinterpret_cast<int*>(ms.l + ATTN_WARPS * MAXG);
    ms.o = reinterpret_cast<float*>(ms.bad + ATTN_WARPS);
    int* gsm = reinterpret_cast<int*>(ms.o + ATTN_WARPS * o.G * OSTRIDE);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // With a static layout (hybrid) the CTA ranges and the addresses of
    // contiguous Persistent Cache tiles depend on the kernel parameters
    // alone: they are worked out before the dependency wait, while the grid
    // is resident early and its predecessor drains, and the first copies go
    // out right after the wait, ahead of the persist_ids round trip.  Layouts
    // that depend on device data (paged) set up after the wait.
    constexpr bool kEarly = Geo::kStaticLayout;
    if constexpr (!kEarly) {
        // Dependents may start only once this grid has passed its own wait,
        // so a dependent's code before its wait sees everything written
        // before this kernel (the merge kernel runs a fused lookup there).
        pdl_wait();
        pdl_launch_dependents();
        geo.cta_init(gsm, o.err_flag, blockIdx.x == 0);
        __syncthreads();
    }

    // Every part is cut into C_p = min(C, tiles of the part) equal ranges;
    // CTA c owns range c of every part (the paged tile count is only known on
    // the device).  No CTA owns an empty range of a part it takes part in,
    // which the partial merge relies on.
    const int C = gridDim.x;
    long long ra[Geo::kParts], rl[Geo::kParts];
    long long total = 0;
#pragma unroll
    for (int p = 0; p < Geo::kParts; ++p) {
        const long long np = geo.part_tiles(p, gsm);
        const long long cp = min(static_cast<long long>(C), np);
        ra[p] = geo.part_begin(p, gsm);
        rl[p] = 0;
        if (static_cast<long long>(blockIdx.x) < cp) {
            ra[p] += np * blockIdx.x / cp;
            rl[p] = geo.part_begin(p, gsm) + np * (blockIdx.x + 1) / cp - ra[p];
        }
        total += rl[p];
    }
    if (!kEarly && total == 0) return;  // uniform over the CTA
    // Odd CTAs take their two ranges in the opposite order, so that half the
    // grid reads scattered Cache Buffer rows while the other half streams
    // the Persistent Cache: the part switch is not taken by every CTA at
    // once (a grid-wide switch stalls the memory pipeline while every warp
    // flushes its segment and waits on its first scattered tile).
    const int pf = (Geo::kParts > 1 && CLO_ATTN_REVERSE_ODD && (blockIdx.x & 1)) ? 1 : 0;
    const int ps = Geo::kParts - 1 - pf;
    // Warp w takes the CTA's tiles w, w + ATTN_WARPS, ... of the concatenated ranges.
    auto tile_at = [&](long long u) -> long long {
        return u < rl[pf] ? ra[pf] + u : ra[ps] + (u - rl[pf]);
    };
    const int nj = warp < total ? static_cast<int>((total - warp + ATTN_WARPS - 1) / ATTN_WARPS) : 0;
    const uint32_t ring = smem_u32(smem) + warp * ATTN_STAGES * STAGE_BYTES;
    uint32_t* my_masks = masks + warp * ATTN_STAGES;

    const uint64_t kv_policy = l2_evict_first_policy();
    Cursor cur;
    bool switched = false;
    Pending pd;
    auto prefetch = [&](int j) {
        const long long u = warp + static_cast<long long>(j) * ATTN_WARPS;
        const long long t = tile_at(u);
        if (Geo::kParts > 1 && u >= rl[pf] && !switched) {
            cursor_init(geo, gsm, t, cur);  // jump to this CTA's range of the other part
            switched = true;
        }
        prefetch_tile(geo, gsm, t, lane, cur, pd);
    };
    const long long u_first = min(static_cast<long long>(warp), total - 1);
    int n_early = 0;
    if constexpr (kEarly) {
        // The first tile of a CTA that starts on the Persistent Cache needs no
        // device data.  Its copies are issued by one code path run twice:
        // before the wait as zero-fill copies (no global reads; this brings
        // the code and the parameters on chip while the predecessor drains),
        // then for real once the wait has passed.
        const bool early = pf == 0 && warp < rl[0] && ATTN_STAGES > 1;  // warp < rl[0]: nj > 0
        if (early) {
            cursor_init(geo, gsm, tile_at(u_first), cur);  // part 0: the table's kv is not used
            prefetch(0);
        }
        int ids_pre = 0;
#pragma unroll 1
        for (int pass = 0; pass < 2; ++pass) {
            if (pass == 1) {
                pdl_wait();  // dependents start only after this (see the paged branch above)
                pdl_launch_dependents();
                if (total == 0) return;  // uniform over the CTA
                ids_pre = geo.ids_preload();
                // A CTA that starts on the Cache Buffer waits two round trips
                // (persist_ids, then its indices) before its first copies, while
                // the DRAM has room.  It uses them to bring the first tiles of
                // its Persistent Cache range into L2; it reads them from there
                // when it gets to them.
                if (Geo::kParts > 1 && pf == 1 && rl[0] > 0 && CLO_ATTN_EARLY_L2_TILES > 0)
                    geo.prefetch_persistent(ra[0], min(rl[0], static_cast<long long>(CLO_ATTN_EARLY_L2_TILES)));
            }
            if (early) {
                issue_tile(geo, gsm, pd, ring, my_masks, lane, kv_policy, pass == 0);
                cp_async_commit();
            }
            if (pass == 0) cp_async_wait<0>();
        }
        n_early = early ? 1 : 0;
        geo.cta_init_with(gsm, o.err_flag, blockIdx.x == 0, ids_pre);
        __syncthreads();
        // At most 128 tiles (8 KB of indices) a CTA: enough for the ranges of
        // these workloads, and bounded for very long ones.
        if (Geo::kParts > 1 && rl[Geo::kParts - 1] > 0)
            geo.prefetch_indices(gsm, ra[Geo::kParts - 1], min(rl[Geo::kParts - 1], 128ll));
    }
    const bool all_bad = geo.all_bad(gsm);
    if (n_early == 0) {
        cursor_init(geo, gsm, tile_at(u_first), cur);
        switched = Geo::kParts > 1 && u_first >= rl[pf];
    }
#pragma unroll
    for (int j = 0; j < ATTN_STAGES - 1; ++j) {
        if (j >= n_early) {
            if (j < nj) {
                prefetch(j);
                issue_tile(geo, gsm, pd, ring + j * STAGE_BYTES, my_masks + j, lane, kv_policy);
            }
            cp_async_commit();
        }
    }
    if (ATTN_STAGES - 1 < nj) prefetch(ATTN_STAGES - 1);

    int jc = 0;
    // ahead: the copies of tile jc + 1 went out before a segment flush (see below).
    bool ahead = false;
    WarpState w;
#pragma unroll 1
    for (int pi = 0; pi < Geo::kParts; ++pi) {
        const int p = pi == 0 ? pf : ps;
        if (rl[p] == 0) continue;
        const long long c0 = ra[p], c1 = ra[p] + rl[p];
        const int s_first = geo.seg_of(c0, gsm), s_last = geo.seg_of(c1 - 1, gsm);
        for (int s = s_first; s <= s_last; ++s) {
            const Seg sg = geo.segment(s, gsm);
            if (sg.ntiles == 0) continue;  // empty requests are zeroed by a separate kernel
            const long long seg_end = sg.first + sg.ntiles;
            uint32_t qb[8][2];
            load_q(o, sg, lane, qb);
            state_reset(w);
            while (jc < nj) {
                const long long t = tile_at(warp + static_cast<long long>(jc) * ATTN_WARPS);
                if (t >= seg_end || t < sg.first) break;  // (a reversed CTA goes back to part 0)
                if (ahead)
                    cp_async_wait<ATTN_STAGES - 1>();
                else
                    cp_async_wait<ATTN_STAGES - 2>();
                __syncwarp();
                const int jn = jc + ATTN_STAGES - 1;
                if (!ahead) {
                    if (jn < nj)
                        issue_tile(geo, gsm, pd, ring + (jn % ATTN_STAGES) * STAGE_BYTES,
                                   my_masks + jn % ATTN_STAGES, lane, kv_policy);
                    cp_async_commit();
                    if (jn + 1 < nj) prefetch(jn + 1);
                }
                ahead = false;
                const int st = jc % ATTN_STAGES;
                const uint32_t mw = *reinterpret_cast<volatile uint32_t*>(my_masks + st);
                w.bad |= static_cast<int>(mw >> 16);
                compute_tile(ring + st * STAGE_BYTES, mw & 0xffffu, qb, o.scale_log2, w, lane);
                ++jc;
            }
            // The warps reach a segment end up to a few microseconds apart and
            // wait for each other in the flush.  The stage of the tile just
            // computed is free, so with many short token sets (paged) the tile
            // after the one in flight is issued into it first and each waiting
            // warp keeps two tiles on the way.  With a few long sets (hybrid)
            // this measured slower: the extra copies queue ahead of the
            // flush's shared-memory loads.
            if (Geo::kAheadAtFlush && ATTN_STAGES == 2 && !ahead && jc + 1 < nj) {
                __syncwarp();
                const int jn = jc + 1;
                issue_tile(geo, gsm, pd, ring + (jn % ATTN_STAGES) * STAGE_BYTES,
                           my_masks + jn % ATTN_STAGES, lane, kv_policy);
                cp_async_commit();
                if (jn + 1 < nj) prefetch(jn + 1);
                ahead = true;
            }
            flush_segment(o, ms, w, sg, s, c0, c1, blockIdx.x + static_cast<size_t>(p) * C,
                          all_bad, warp, lane);
        }
    }
    cp_async_wait<0>();
}

// Zeroes the outputs of requests with no tokens (paged only).
__global__ void paged_zero_empty_kernel(const int32_t* __restrict__ ctx_len, int B, int max_tok,
                                        int Hq, clo_half* __restrict__ out, float* __restrict__ lse) {
    pdl_launch_dependents();
    pdl_wait();
    const int r = blockIdx.x;
    if (r >= B) return;
    const int n = ctx_len[r];
    if (n > 0 && n <= max_tok) return;
    for (int i = threadIdx.x; i < Hq * D; i += blockDim.x)
        out[static_cast<size_t>(r) * Hq * D + i] = 0;
    if (lse != nullptr)
        for (int h = threadIdx.x; h < Hq; h += blockDim.x)
            lse[static_cast<size_t>(r) * Hq + h] = -INFINITY;
}

// Merges the per-CTA partials of every token set cut by CTA boundaries.  A
// block handles `hpb` query heads of one cut token set (the host picks all G
// heads when every set has few partials, one head per block when some set
// has many).  Thread (group, head, column) folds every ngrp-th partial of 8
// output columns in one online log-sum-exp pass, eight partials per trip with
// independent loads; the groups are then combined in shared memory.
constexpr int MERGE_COLS = 8;                                   // floats per thread and partial
constexpr int MERGE_ITEMS = D / MERGE_COLS;                     // 16 column groups per head
constexpr int MERGE_MAX_GROUPS = MERGE_THREADS / MERGE_ITEMS;   // 32 partial subsets
constexpr int MERGE_UNROLL = 8;                                 // independent partials per trip

template <class Geo>
__global__ void __launch_bounds__(MERGE_THREADS, 1)
    attn_merge_kernel(const Geo geo, const AttnOut o, int C, int hpb, int n_merge,
                      const LookupParams lk, int lk_first) {
    extern __shared__ __align__(16) uint8_t msmem[];
    // Block (x, y) merges query heads [y * hpb, (y + 1) * hpb) of one cut token set.
    const int G = o.G;
    const int items = hpb * MERGE_ITEMS;
    const int ngrp = min(MERGE_THREADS / items, MERGE_MAX_GROUPS);
    float* Mg = reinterpret_cast<float*>(msmem);                     // [ngrp][MAXG]
    float* Lg = Mg + MERGE_MAX_GROUPS * MAXG;                        // [ngrp][MAXG]
    int* Bg = reinterpret_cast<int*>(Lg + MERGE_MAX_GROUPS * MAXG);  // [ngrp][MAXG]
    float4* Og = reinterpret_cast<float4*>(Bg + MERGE_MAX_GROUPS * MAXG);  // [ngrp][items][2]
    int* gsm = reinterpret_cast<int*>(Og + 2 * MERGE_THREADS);

    pdl_launch_dependents();
    if (static_cast<int>(blockIdx.x) >= n_merge) {
        // Past the merge blocks: one cluster at the end of row 0 runs the
        // next layer's lookup; the other blocks only pad the grid to whole
        // clusters.  The lookup reads nothing the attention writes, and the
        // main kernel let this grid start only after its own dependency wait,
        // so it needs no wait of its own and overlaps the main kernel's tail.
        if (lk.B > 0 && static_cast<int>(blockIdx.x) >= lk_first && blockIdx.y == 0) {
            __shared__ int lk_misses;
            lookup_cluster<MERGE_THREADS / 32>(lk, msmem, &lk_misses);
        }
        if (blockIdx.x == 0 && blockIdx.y == 0) pdl_wait();  // see below
        return;
    }
    // Static layouts (hybrid): block s handles token set s if CTA boundaries
    // cut it; the test needs no memory, so blocks with nothing to merge leave
    // at once.  Dynamic layouts (paged): block (part, i) looks at the boundary
    // between CTA ranges i and i + 1 and handles the token set that crosses
    // it if that set starts in range i.  Partial slots of part p are offset by
    // p * C.
    int s, part, c_lo, P;
    if (Geo::kStaticLayout) {
        s = blockIdx.x;
        part = geo.segment_part(s);
        const long long P0 = geo.part_begin(part, nullptr);
        const long long N = geo.part_tiles(part, nullptr);
        const long long Ce = min(static_cast<long long>(C), N);
        const long long first = geo.segment_first(s) - P0;
        const long long last = first + geo.segment_ntiles(s) - 1;
        c_lo = static_cast<int>(((first + 1) * Ce - 1) / N);
        const int c_hi = static_cast<int>(((last + 1) * Ce - 1) / N);
        // Block (0, 0) waits for the grid ahead even with nothing to merge
        // (as do the blocks that merge), so this grid never finishes before
        // that grid, nor, through that grid's own wait, before any kernel
        // further back: the next kernel, which waits for this grid alone,
        // finds all of them finished.  (A fill launched beside the main
        // kernel relies on it: the next layer's attention reads its rows.)
        if (c_lo == c_hi) {
            if (blockIdx.x == 0 && blockIdx.y == 0) pdl_wait();
            return;
        }
        P = c_hi - c_lo + 1;
        pdl_wait();
    } else {
        pdl_wait();
        geo.cta_init(gsm, nullptr, false);
        __syncthreads();
        part = blockIdx.x / (C - 1);
        const int i = blockIdx.x - part * (C - 1);
        const long long P0 = geo.part_begin(part, gsm);
        const long long N = geo.part_tiles(part, gsm);
        const int Ce = static_cast<int>(min(static_cast<long long>(C), N));  // CTAs with a range
        if (i >= Ce - 1) return;
        const long long start_i = P0 + N * i / Ce, tb = P0 + N * (i + 1) / Ce;
        s = geo.seg_of(tb, gsm);
        const long long first = geo.segment(s, gsm).first;
        if (!(first < tb && first >= start_i)) return;
        const long long last = first + geo.segment(s, gsm).ntiles - 1 - P0;
        c_lo = i;
        P = static_cast<int>(((last + 1) * Ce - 1) / N) - i + 1;
    }
    // Output rows of the set: batch row and KV head.  With a static layout
    // the last warp loads persist_ids now and resolves the KV head once its
    // partials are in; it is published before the combine below.
    __shared__ int kv_sm, ids_bad_sm;
    int b_out;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int kIdsWarp = MERGE_THREADS / 32 - 1;
    int id0 = -1, id1 = -1;
    if (Geo::kStaticLayout) {
        b_out = geo.segment(s, nullptr, true).b;
        if constexpr (Geo::kStaticLayout)
            if (warp == kIdsWarp) geo.ids_warp_load(lane, id0, id1);
    } else {
        const Seg sg0 = geo.segment(s, gsm);
        b_out = sg0.b;
        if (threadIdx.x == 0) {
            kv_sm = sg0.kv;
            ids_bad_sm = 0;
        }
    }
    const size_t slot0 = static_cast<size_t>(c_lo) + static_cast<size_t>(s) +
                         static_cast<size_t>(part) * C;

    const int it = threadIdx.x % items, grp = threadIdx.x / items;
    const int hl = it / MERGE_ITEMS, col = it % MERGE_ITEMS;  // head within the block, column
    const int h = blockIdx.y * hpb + hl;
    float M = -INFINITY, L = 0.f;
    float a[MERGE_COLS];
#pragma unroll
    for (int c = 0; c < MERGE_COLS; ++c) a[c] = 0.f;
    int bad = 0;
    if (grp < ngrp) {
        for (int p0 = grp; p0 < P; p0 += MERGE_UNROLL * ngrp) {
            float x[MERGE_UNROLL];
            float4 v0[MERGE_UNROLL], v1[MERGE_UNROLL];
#pragma unroll
            for (int u = 0; u < MERGE_UNROLL; ++u) {
                const int p = p0 + u * ngrp;
                x[u] = -INFINITY;
                v0[u] = v1[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (p < P) {
                    const size_t slot = slot0 + p;
                    x[u] = o.ws_lse[slot * G + h];
                    const float4* src =
                        reinterpret_cast<const float4*>(o.ws_o + (slot * G + h) * D) + 2 * col;
                    v0[u] = src[0];
                    v1[u] = src[1];
                }
            }
            float mx = M;
#pragma unroll
            for (int u = 0; u < MERGE_UNROLL; ++u) {
                if (x[u] == INFINITY) {
                    bad = 1;
                    x[u] = -INFINITY;
                }
                mx = fmaxf(mx, x[u]);
            }
            if (mx == -INFINITY) continue;
            const float sc = fast_exp2(M - mx);
            L *= sc;
#pragma unroll
            for (int c = 0; c < MERGE_COLS; ++c) a[c] *= sc;
#pragma unroll
            for (int u = 0; u < MERGE_UNROLL; ++u) {
                const float e = fast_exp2(x[u] - mx);
                L += e;
                a[0] = fmaf(v0[u].x, e, a[0]);
                a[1] = fmaf(v0[u].y, e, a[1]);
                a[2] = fmaf(v0[u].z, e, a[2]);
                a[3] = fmaf(v0[u].w, e, a[3]);
                a[4] = fmaf(v1[u].x, e, a[4]);
                a[5] = fmaf(v1[u].y, e, a[5]);
                a[6] = fmaf(v1[u].z, e, a[6]);
                a[7] = fmaf(v1[u].w, e, a[7]);
            }
            M = mx;
        }
        if (col == 0) {
            Mg[grp * MAXG + hl] = M;
            Lg[grp * MAXG + hl] = L;
            Bg[grp * MAXG + hl] = bad;
        }
        Og[2 * (grp * items + it)] = make_float4(a[0], a[1], a[2], a[3]);
        Og[2 * (grp * items + it) + 1] = make_float4(a[4], a[5], a[6], a[7]);
    }
    if constexpr (Geo::kStaticLayout) {
        if (warp == kIdsWarp) {
            bool ids_ok;
            const int kv = geo.segment_kv_warp(s, lane, id0, id1, ids_ok);
            if (lane == 0) {
                kv_sm = kv;
                ids_bad_sm = ids_ok ? 0 : 1;
            }
        }
    }
    __syncthreads();
    // Tree over the thread groups: at each level group g < n - half takes in
    // group g + half (a fixed order, so the result does not depend on timing).
    for (int n = ngrp; n > 1;) {
        const int half = (n + 1) >> 1;
        if (grp < n - half) {
            const int q2 = grp + half;
            const float m2 = Mg[q2 * MAXG + hl];
            bad |= Bg[q2 * MAXG + hl];
            const float mx = fmaxf(M, m2);
            if (mx != -INFINITY) {
                const float e1 = fast_exp2(M - mx), e2 = fast_exp2(m2 - mx);
                const float4 w0 = Og[2 * (q2 * items + it)], w1 = Og[2 * (q2 * items + it) + 1];
                L = L * e1 + Lg[q2 * MAXG + hl] * e2;
                a[0] = fmaf(w0.x, e2, a[0] * e1);
                a[1] = fmaf(w0.y, e2, a[1] * e1);
                a[2] = fmaf(w0.z, e2, a[2] * e1);
                a[3] = fmaf(w0.w, e2, a[3] * e1);
                a[4] = fmaf(w1.x, e2, a[4] * e1);
                a[5] = fmaf(w1.y, e2, a[5] * e1);
                a[6] = fmaf(w1.z, e2, a[6] * e1);
                a[7] = fmaf(w1.w, e2, a[7] * e1);
                M = mx;
            }
            if (half > 1) {
                if (col == 0) {
                    Mg[grp * MAXG + hl] = M;
                    Lg[grp * MAXG + hl] = L;
                    Bg[grp * MAXG + hl] = bad;
                }
                Og[2 * (grp * items + it)] = make_float4(a[0], a[1], a[2], a[3]);
                Og[2 * (grp * items + it) + 1] = make_float4(a[4], a[5], a[6], a[7]);
            }
        }
        __syncthreads();
        n = half;
    }
    if (grp == 0) {
        bad |= ids_bad_sm;
        const bool empty = !(L > 0.f);
        const size_t row = static_cast<size_t>(b_out) * o.Hq + static_cast<size_t>(kv_sm) * G + h;
        const float inv = (bad || empty) ? 0.f : 1.f / L;
        uint4 pk;
        __half2 h0 = __floats2half2_rn(a[0] * inv, a[1] * inv);
        __half2 h1 = __floats2half2_rn(a[2] * inv, a[3] * inv);
        __half2 h2 = __floats2half2_rn(a[4] * inv, a[5] * inv);
        __half2 h3 = __floats2half2_rn(a[6] * inv, a[7] * inv);
        pk.x = *reinterpret_cast<uint32_t*>(&h0);
        pk.y = *reinterpret_cast<uint32_t*>(&h1);
        pk.z = *reinterpret_cast<uint32_t*>(&h2);
        pk.w = *reinterpret_cast<uint32_t*>(&h3);
        reinterpret_cast<uint4*>(o.out + row * D)[col] = pk;
        if (o.lse != nullptr && col == 0)
            o.lse[row] = (bad || empty) ? -INFINITY : (M + log2f(L)) * LN2;
    }
}

// ---------------------------------------------------------------- host side

static bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Bytes of the split-KV partials: [slots][G][128] fp32 outputs, then
// [slots][G] fp32 log2-sum-exps, each padded to 256 bytes.
static size_t partial_bytes(long long slots, int G) {
    const size_t o = static_cast<size_t>(slots) * G * D * sizeof(float);
    const size_t l = static_cast<size_t>(slots) * G * sizeof(float);
    return ((o + 255) / 256) * 256 + ((l + 255) / 256) * 256;
}

static size_t workspace_bytes(int B, int Hq, int Hkv, int d, int num_ctas) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d != D || num_ctas < 0) return 0;
    const int G = Hq / Hkv;
    if (G > MAXG) return 0;
    int C = num_ctas > 0 ? num_ctas : device_sm_count() * ATTN_CTAS_PER_SM;
    if (C <= 0) return 0;
    return partial_bytes(2ll * C + static_cast<long long>(B) * Hkv, G);
}

static size_t attn_smem_bytes(int G, size_t geo_ints) {
    return static_cast<size_t>(ATTN_WARPS) * ATTN_STAGES * STAGE_BYTES +
           ATTN_WARPS * ATTN_STAGES * sizeof(uint32_t) + 2 * ATTN_WARPS * MAXG * sizeof(float) +
           ATTN_WARPS * sizeof(int) + static_cast<size_t>(ATTN_WARPS) * G * OSTRIDE * sizeof(float) +
           geo_ints * sizeof(int);
}

static size_t merge_smem_bytes(int /*G*/, size_t geo_ints) {
    return static_cast<size_t>(MERGE_MAX_GROUPS) * MAXG * 3 * sizeof(float) +
           static_cast<size_t>(2) * MERGE_THREADS * sizeof(float4) + geo_ints * sizeof(int);
}

// Launches the main kernel, then (if given) a fill beside it, then the merge
// launch (carrying the lookup, if given).
template <class Geo>
static clo_status launch_attention(const Geo& geo, AttnOut o, long long n_tiles_host_bound,
                                   size_t geo_ints, int S, void* workspace, size_t ws_bytes,
                                   const clo_attn_opts* opts, cudaStream_t stream,
                                   const LookupParams* lookup = nullptr,
                                   const FillParams* fill = nullptr, int fill_ctas = 0) {
    if (!prepare_kernel(reinterpret_cast<const void*>(attn_split_kernel<Geo>), SMEM_LIMIT) ||
        !prepare_kernel(reinterpret_cast<const void*>(attn_merge_kernel<Geo>), MERGE_SMEM_LIMIT))
        return CLO_ERR_CUDA;
    const size_t smem = attn_smem_bytes(o.G, geo_ints);
    const size_t msmem = merge_smem_bytes(o.G, geo_ints);
    if (smem > static_cast<size_t>(SMEM_LIMIT) || msmem > static_cast<size_t>(MERGE_SMEM_LIMIT))
        return CLO_ERR_UNSUPPORTED;

    // As many CTAs per SM as fit, at most ATTN_CTAS_PER_SM (a large query
    // group needs a larger merge area).
    int per_sm = static_cast<int>(SMEM_PER_SM / (smem + 1024));
    if (per_sm > ATTN_CTAS_PER_SM) per_sm = ATTN_CTAS_PER_SM;
    if (per_sm < 1) return CLO_ERR_UNSUPPORTED;
    const int wave = device_sm_count() * per_sm;
    if (wave <= 0) return CLO_ERR_CUDA;
    // A fill carried beside the main kernel runs in CTA slots the main grid
    // leaves free (a fill CTA fits in the room of one main-kernel CTA).
    long long fill_grid = 0;
    if (fill != nullptr) {
        fill_grid = fill_ctas > 0 ? fill_ctas : fill_beside_default_ctas(*fill, wave);
        if (fill_grid <= 0) return CLO_ERR_CUDA;
    }
    int C = (opts != nullptr && opts->num_ctas > 0)
                ? opts->num_ctas
                : static_cast<int>(std::max(wave - fill_grid, 1ll));
    // Never more CTAs than tiles (no CTA gets an empty range) and at least one
    // tile per warp where the problem allows.
    const long long cap = n_tiles_host_bound / ATTN_WARPS;
    if (C > cap) C = static_cast<int>(cap > 0 ? cap : 1);
    if (C > n_tiles_host_bound) C = static_cast<int>(n_tiles_host_bound);
    if (C < 1) C = 1;
    const long long slots = 2ll * C + S;  // room for one partial per (part, CTA, segment)
    const size_t need = partial_bytes(slots, o.G);
    if (workspace == nullptr || ws_bytes < need || !aligned(workspace, 16)) return CLO_ERR_WORKSPACE;
    o.ws_o = static_cast<float*>(workspace);
    o.ws_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                        ((static_cast<size_t>(slots) * o.G * D * sizeof(float) + 255) / 256) * 256);

    if (opts != nullptr && opts->ev_begin != nullptr && !record_event(opts->ev_begin, stream))
        return CLO_ERR_CUDA;
    if (launch_pdl(attn_split_kernel<Geo>, dim3(C), dim3(ATTN_THREADS), smem, stream, geo, o) !=
        cudaSuccess)
        return CLO_ERR_CUDA;
    // The fill starts as soon as every main-kernel CTA has passed its
    // dependency wait and runs beside them; the launches below wait for it,
    // and it waits for the main kernel at its end.
    if (fill != nullptr &&
        launch_fill(*fill, static_cast<int>(fill_grid), true, stream) != cudaSuccess)
        return CLO_ERR_CUDA;
    if (opts != nullptr && opts->ev_end != nullptr && !record_event(opts->ev_end, stream))
        return CLO_ERR_CUDA;
    const int merge_blocks =
        C < 2 ? 0 : (Geo::kStaticLayout ? geo.num_segments() : Geo::kParts * (C - 1));
    // All heads in one block when every cut token set has few enough partials
    // for one round of loads per thread group; else one head per block.
    int hpb = o.G;
    if (C >= 2) {
        const long long most = geo.max_partials_host(C);
        const int ngrp_all = MERGE_THREADS / (o.G * MERGE_ITEMS);
        hpb = most <= static_cast<long long>(ngrp_all) * MERGE_UNROLL ? o.G : 1;
    }
    // A large lookup runs beside the main kernel's drain, launched after it
    // (and after the fill, whose CTAs start first); the merge launch then
    // carries nothing else.  A small one rides in the merge launch (below).
    if (lookup != nullptr &&
        static_cast<long long>(lookup->B) * lookup->Hkv >= LK_BESIDE_MIN_GROUPS) {
        if (launch_lookup_beside(*lookup, stream) != cudaSuccess) return CLO_ERR_CUDA;
        lookup = nullptr;
    }
    LookupParams none{};
    if (lookup == nullptr) {
        if (merge_blocks > 0 &&
            launch_pdl(attn_merge_kernel<Geo>, dim3(merge_blocks, o.G / hpb), dim3(MERGE_THREADS),
                       msmem, stream, geo, o, C, hpb, merge_blocks, none, merge_blocks) !=
                cudaSuccess)
            return CLO_ERR_CUDA;
        return CLO_OK;
    }
    // The next layer's lookup rides in the merge launch: whole clusters of
    // LK_CLUSTER blocks, the lookup's cluster last.
    const int lk_first = (merge_blocks + LK_CLUSTER - 1) / LK_CLUSTER * LK_CLUSTER;
    const size_t lsmem = std::max(msmem, static_cast<size_t>(lookup_smem_bytes(lookup->B, lookup->Hkv)));
    if (lsmem > static_cast<size_t>(MERGE_SMEM_LIMIT)) return CLO_ERR_UNSUPPORTED;
    if (launch_pdl_cluster(attn_merge_kernel<Geo>, dim3(lk_first + LK_CLUSTER, o.G / hpb),
                           dim3(MERGE_THREADS), lsmem, stream, LK_CLUSTER, geo, o, C, hpb,
                           merge_blocks, *lookup, lk_first) != cudaSuccess)
        return CLO_ERR_CUDA;
    return CLO_OK;
}

}  // namespace clo

using namespace clo;

extern "C" size_t clo_hybrid_workspace_size(int B, int Hq, int Hkv, int d, int num_ctas) {
    return workspace_bytes(B, Hq, Hkv, d, num_ctas);
}

extern "C" size_t clo_paged_workspace_size(int B, int Hq, int Hkv, int d, int num_ctas) {
    return workspace_bytes(B, Hq, Hkv, d, num_ctas);
}

static clo_status hybrid_attention(const clo_half* q, const clo_half* cbK, const clo_half* cbV,
                                   const int32_t* idx, int k, int C, const clo_half* pK,
                                   const clo_half* pV, const int32_t* persist_ids, int Np, int T,
                                   int B, int Hq, int Hkv, int d, float scale, clo_half* out,
                                   float* lse, void* workspace, size_t ws_bytes, int32_t* err_flag,
                                   const clo_attn_opts* opts, cudaStream_t stream,
                                   const LookupParams* lookup, const FillParams* fill = nullptr,
                                   int fill_ctas = 0) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || Np < 0 || Np > Hkv)
        return CLO_ERR_INVALID_ARG;
    if (B == 0) return CLO_OK;  // empty batch: nothing to compute
    if (q == nullptr || out == nullptr) return CLO_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !isfinite(scale)) return CLO_ERR_INVALID_ARG;
    const int G = Hq / Hkv;
    if (d != D || G > MAXG || Hkv > MAX_HKV_HYBRID) return CLO_ERR_UNSUPPORTED;
    const bool has_cb = Np < Hkv;
    if (C > MAX_ROWS || T > MAX_ROWS) return CLO_ERR_UNSUPPORTED;
    if (has_cb) {
        if (cbK == nullptr || cbV == nullptr || idx == nullptr || k < 1 || C < k)
            return CLO_ERR_INVALID_ARG;
        if (!aligned(cbK, 16) || !aligned(cbV, 16) || !aligned(idx, 4)) return CLO_ERR_INVALID_ARG;
    }
    if (Np > 0) {
        if (pK == nullptr || pV == nullptr || persist_ids == nullptr || T < 1)
            return CLO_ERR_INVALID_ARG;
        if (!aligned(pK, 16) || !aligned(pV, 16) || !aligned(persist_ids, 4))
            return CLO_ERR_INVALID_ARG;
    }
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(lse, 4)) return CLO_ERR_INVALID_ARG;

    HybridGeo geo;
    geo.cbK = cbK;
    geo.cbV = cbV;
    geo.idx = idx;
    geo.pK = pK;
    geo.pV = pV;
    geo.persist_ids = persist_ids;
    geo.k = has_cb ? k : 0;
    geo.C = has_cb ? C : 0;
    geo.Np = Np;
    geo.T = Np > 0 ? T : 0;
    geo.B = B;
    geo.Hkv = Hkv;
    geo.tp = Np > 0 ? (T + TILE - 1) / TILE : 1;
    geo.tc = has_cb ? (k + TILE - 1) / TILE : 1;
    geo.n0 = static_cast<long long>(B) * Np * (Np > 0 ? geo.tp : 0);
    geo.n1 = static_cast<long long>(B) * (Hkv - Np) * (has_cb ? geo.tc : 0);
    const long long N = geo.n0 + geo.n1;
    if (N >= (1ll << 31)) return CLO_ERR_UNSUPPORTED;  // tile counts stay 32-bit per CTA

    AttnOut o{};
    o.q = q;
    o.out = out;
    o.lse = lse;
    o.err_flag = err_flag;
    o.scale_log2 = scale * LOG2E;
    o.Hq = Hq;
    o.G = G;
    return launch_attention(geo, o, N, HybridGeo::smem_ints(Hkv, B), B * Hkv, workspace,
                            ws_bytes, opts, stream, lookup, fill, fill_ctas);
}

extern "C" clo_status clo_hybrid_decode_attn(const clo_half* q, const clo_half* cbK,
                                             const clo_half* cbV, const int32_t* idx, int k, int C,
                                             const clo_half* pK, const clo_half* pV,
                                             const int32_t* persist_ids, int Np, int T, int B,
                                             int Hq, int Hkv, int d, float scale, clo_half* out,
                                             float* lse, void* workspace, size_t ws_bytes,
                                             int32_t* err_flag, const clo_attn_opts* opts,
                                             cudaStream_t stream) {
    return hybrid_attention(q, cbK, cbV, idx, k, C, pK, pV, persist_ids, Np, T, B, Hq, Hkv, d,
                            scale, out, lse, workspace, ws_bytes, err_flag, opts, stream, nullptr);
}

extern "C" clo_status clo_hybrid_decode_attn_lookup(
    const clo_half* q, const clo_half* cbK, const clo_half* cbV, const int32_t* idx, int k, int C,
    const clo_half* pK, const clo_half* pV, const int32_t* persist_ids, int Np, int T, int B,
    int Hq, int Hkv, int d, float scale, clo_half* out, float* lse, void* workspace,
    size_t ws_bytes, int32_t* err_flag, const clo_half* q_next, clo_half* labels_next,
    const float* w_q_next, const float* tau_next, const uint8_t* persist_mask_next,
    uint8_t* flag_next, float* sim_next, int32_t* miss_list_next, int32_t* miss_count_next,
    const clo_attn_opts* opts, cudaStream_t stream) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return CLO_ERR_INVALID_ARG;
    if (miss_count_next == nullptr || !aligned(miss_count_next, 4)) return CLO_ERR_INVALID_ARG;
    if (B == 0)  // nothing to attend to or look up: only the miss count is written
        return cudaMemsetAsync(miss_count_next, 0, sizeof(int32_t), stream) == cudaSuccess
                   ? CLO_OK
                   : CLO_ERR_CUDA;
    LookupParams lk;
    const clo_status st = make_lookup_params(q_next, labels_next, w_q_next, tau_next,
                                             persist_mask_next, B, Hq, Hkv, d, flag_next,
                                             sim_next, miss_list_next, miss_count_next, lk);
    if (st != CLO_OK) return st;
    return hybrid_attention(q, cbK, cbV, idx, k, C, pK, pV, persist_ids, Np, T, B, Hq, Hkv, d,
                            scale, out, lse, workspace, ws_bytes, err_flag, opts, stream, &lk);
}

extern "C" clo_status clo_hybrid_decode_layer(
    const clo_half* q, const clo_half* cbK, const clo_half* cbV, const int32_t* idx, int k, int C,
    const clo_half* pK, const clo_half* pV, const int32_t* persist_ids, int Np, int T, int B,
    int Hq, int Hkv, int d, float scale, clo_half* out, float* lse, void* workspace,
    size_t ws_bytes, int32_t* err_flag, const clo_fill_args* fill, const clo_lookup_args* lookup,
    const clo_attn_opts* opts, cudaStream_t stream) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return CLO_ERR_INVALID_ARG;
    if (fill != nullptr && fill->num_ctas < 0) return CLO_ERR_INVALID_ARG;
    LookupParams lk;
    if (lookup != nullptr) {
        if (lookup->miss_count == nullptr || !aligned(lookup->miss_count, 4))
            return CLO_ERR_INVALID_ARG;
        if (B > 0) {
            const clo_status st = make_lookup_params(
                lookup->q, lookup->labels, lookup->w_q, lookup->tau, lookup->persist_mask, B, Hq,
                Hkv, d, lookup->flag, lookup->sim, lookup->miss_list, lookup->miss_count, lk);
            if (st != CLO_OK) return st;
        }
    }
    FillParams fp;
    bool no_fill = true;
    if (fill != nullptr) {
        const clo_status st = make_fill_params(fill->srcK, fill->srcV, fill->T, fill->tok,
                                               fill->slot, fill->k, fill->cbK, fill->cbV, fill->C,
                                               fill->miss_list, fill->miss_count, B, Hkv, d,
                                               err_flag, fp, no_fill);
        if (st != CLO_OK) return st;
        // The fill runs beside this layer's attention and the lookup carried
        // after it: it must not write what the attention reads, nor read the
        // miss list the lookup writes.
        if (!no_fill && ((cbK != nullptr && fill->cbK == cbK) || (cbV != nullptr && fill->cbV == cbV)))
            return CLO_ERR_INVALID_ARG;
        if (!no_fill && lookup != nullptr &&
            (fill->miss_list == lookup->miss_list || fill->miss_count == lookup->miss_count))
            return CLO_ERR_INVALID_ARG;
    }
    if (B == 0)  // nothing to attend to, fill or look up: only a lookup's miss count is written
        return lookup == nullptr || cudaMemsetAsync(lookup->miss_count, 0, sizeof(int32_t),
                                                    stream) == cudaSuccess
                   ? CLO_OK
                   : CLO_ERR_CUDA;
    return hybrid_attention(q, cbK, cbV, idx, k, C, pK, pV, persist_ids, Np, T, B, Hq, Hkv, d,
                            scale, out, lse, workspace, ws_bytes, err_flag, opts, stream,
                            lookup != nullptr ? &lk : nullptr, no_fill ? nullptr : &fp,
                            fill != nullptr ? fill->num_ctas : 0);
}

extern "C" clo_status clo_paged_decode_attn(const clo_half* q, const clo_half* kc,
                                            const clo_half* vc, const int32_t* block_table,
                                            int max_blocks, const int32_t* ctx_len,
                                            int num_blocks, int B, int Hq, int Hkv, int d,
                                            int block_size, float scale, clo_half* out, float* lse,
                                            void* workspace, size_t ws_bytes, int32_t* err_flag,
                                            const clo_attn_opts* opts, cudaStream_t stream) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || max_blocks < 1 || num_blocks < 1)
        return CLO_ERR_INVALID_ARG;
    if (B == 0) return CLO_OK;  // no requests: nothing to compute
    if (q == nullptr || kc == nullptr || vc == nullptr || block_table == nullptr ||
        ctx_len == nullptr || out == nullptr)
        return CLO_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !isfinite(scale)) return CLO_ERR_INVALID_ARG;
    const int G = Hq / Hkv;
    if (d != D || G > MAXG || block_size != TILE || B > MAX_PAGED_B) return CLO_ERR_UNSUPPORTED;
    if (static_cast<long long>(B) * Hkv * max_blocks >= (1ll << 31)) return CLO_ERR_UNSUPPORTED;
    if (!aligned(q, 16) || !aligned(kc, 16) || !aligned(vc, 16) || !aligned(out, 16) ||
        !aligned(block_table, 4) || !aligned(ctx_len, 4) || !aligned(lse, 4))
        return CLO_ERR_INVALID_ARG;

    PagedGeo geo;
    geo.kc = kc;
    geo.vc = vc;
    geo.block_table = block_table;
    geo.ctx_len = ctx_len;
    geo.max_blocks = max_blocks;
    geo.num_blocks = num_blocks;
    geo.B = B;
    geo.Hkv = Hkv;

    AttnOut o{};
    o.q = q;
    o.out = out;
    o.lse = lse;
    o.err_flag = err_flag;
    o.scale_log2 = scale * LOG2E;
    o.Hq = Hq;
    o.G = G;
    // Requests with no tokens (or an invalid length) get zeros before the main kernel.
    if (!prepare_kernel(reinterpret_cast<const void*>(paged_zero_empty_kernel), 0))
        return CLO_ERR_CUDA;
    if (launch_pdl(paged_zero_empty_kernel, dim3(B), dim3(128), 0, stream, ctx_len, B,
                   max_blocks * TILE, Hq, out, lse) != cudaSuccess)
        return CLO_ERR_CUDA;
    // The tile count depends on device-resident lengths; size the grid for the
    // largest possible stream (CTAs never exceed the true count, see kernel).
    const long long bound = static_cast<long long>(B) * Hkv * max_blocks;
    return launch_attention(geo, o, bound, PagedGeo::smem_ints(Hkv, B), B * Hkv, workspace,
                            ws_bytes, opts, stream);
}

// ---------------------------------------------------------------- no-allocation variant
// Some callers cannot allocate device memory when they run this path: serving
// engines that hand every free byte of the GPU to their own pool at start-up
// and forbid outside allocations, deployments that freeze allocation after
// start-up, and host programs that reach the library through its C ABI alone,
// with no allocator of their own.  clo_hybrid_decode_attn_noalloc serves
// them: its split-KV scratch is the fixed array below, part of the library
// image, which every GPU that loads the library keeps until the process exits.
namespace clo {
constexpr size_t NOALLOC_SCRATCH_BYTES = size_t(8) << 20;  // 8 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// with the device current, once per device and context, then cached; a new
// context on the device (after cudaDeviceReset) is looked up again.
static void* noalloc_scratch_address() {
    static std::mutex mu;
    static void* addr[64] = {nullptr};
    static unsigned long long ctx_of[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lock(mu);
    if (ctx != 0 && addr[dev] != nullptr && ctx_of[dev] == ctx) return addr[dev];
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    addr[dev] = p;
    ctx_of[dev] = current_context_id();  // the lookup made the primary context current
    return p;
}
}  // namespace clo

extern "C" size_t clo_hybrid_noalloc_max_scratch(void) { return clo::NOALLOC_SCRATCH_BYTES; }

extern "C" clo_status clo_hybrid_decode_attn_noalloc(
    const clo_half* q, const clo_half* cbK, const clo_half* cbV, const int32_t* idx, int k, int C,
    const clo_half* pK, const clo_half* pV, const int32_t* persist_ids, int Np, int T, int B,
    int Hq, int Hkv, int d, float scale, clo_half* out, float* lse, int32_t* err_flag,
    const clo_attn_opts* opts, cudaStream_t stream) {
    if (B == 0)
        return clo_hybrid_decode_attn(q, cbK, cbV, idx, k, C, pK, pV, persist_ids, Np, T, B, Hq,
                                      Hkv, d, scale, out, lse, nullptr, 0, err_flag, opts, stream);
    const int num_ctas = opts != nullptr ? opts->num_ctas : 0;
    const size_t need = clo_hybrid_workspace_size(B, Hq, Hkv, d, num_ctas);
    if (need > clo::NOALLOC_SCRATCH_BYTES) return CLO_ERR_WORKSPACE;  // problem too large
    void* scratch = clo::noalloc_scratch_address();
    if (scratch == nullptr) return CLO_ERR_CUDA;
    return clo_hybrid_decode_attn(q, cbK, cbV, idx, k, C, pK, pV, persist_ids, Np, T, B, Hq, Hkv,
                                  d, scale, out, lse, scratch, clo::NOALLOC_SCRATCH_BYTES,
                                  err_flag, opts, stream);
}
