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
//    one KV head).  All tiles of all segments form one flat stream, which is
//    cut into C equal contiguous ranges, one per CTA (C = SM count).  Every SM
//    therefore streams the same number of KV bytes whether a tile comes from a
//    128K-token persistent head or from a 13K-row top-k head -- the few long
//    persistent heads cannot serialise the launch.
//  * Inside a CTA the 8 warps take the range's tiles round-robin.  Each warp
//    keeps its own 3-stage shared-memory ring filled by 16-byte cp.async
//    copies (K and V rows of a tile: 8 KB), so ~128 KB per SM is in flight.
//    Rows are XOR-swizzled in 16-byte chunks so ldmatrix reads are bank-
//    conflict free.  Indexed rows (Cache Buffer) and block-table rows cost the
//    same as contiguous rows: every copy is a whole 256-byte row.
//  * Math on the tensor cores with mma.sync m16n8k16 (fp16 in, fp32 accum):
//    S = K_tile Q^T puts the 16 tokens on M and the G <= 8 query heads of the
//    KV group on N (one n8 tile), then O^T += V_tile^T P^T puts the 128 head
//    dimensions on M and the heads on N.  P is moved from the S accumulator
//    layout to the B-operand layout with movmatrix.trans.  Online softmax in
//    the exp2 domain with per-tile warp-shuffle max.
//  * Each CTA merges its warps' (m, l, O) in shared memory whenever its range
//    crosses a segment end.  A segment that lies wholly in one CTA is written
//    straight to the output; a segment cut by CTA boundaries leaves one fp32
//    partial per CTA in the workspace (slot c + s, unique because both
//    partitions are contiguous) and a second small kernel merges those
//    partials by log-sum-exp.
//  * Bad indices, block-table entries, context lengths or persistent ids are
//    never dereferenced: the copy is zero-filled, the row masked, an error bit
//    is ORed into err_flag and the affected outputs are written as zeros.
#include <math.h>

#include <mutex>

#include "clo_device.cuh"

namespace clo {

constexpr int D = 128;
constexpr int TILE = 16;
constexpr int ROW_BYTES = D * 2;
constexpr int KV_TILE_BYTES = TILE * ROW_BYTES;  // 4 KB of K (or V) per tile
constexpr int STAGE_BYTES = 2 * KV_TILE_BYTES;   // K + V
constexpr int MAXG = 8;
constexpr int OSTRIDE = D + 4;  // padded merge-area row (floats): conflict-free writes
constexpr int ATTN_WARPS = 8;
constexpr int ATTN_STAGES = 3;
constexpr int ATTN_THREADS = ATTN_WARPS * 32;
constexpr int MERGE_THREADS = 1024;
constexpr int MAX_HKV_HYBRID = 64;
constexpr int MAX_PAGED_B = 4096;
constexpr int SMEM_LIMIT = 227 * 1024;

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
// Segments are ordered (b, slot): slots [0, Np) are the persistent heads in
// persist_ids order (T tokens each), slots [Np, Hkv) the remaining KV heads in
// ascending order (k indexed Cache Buffer rows each).
struct HybridGeo {
    const clo_half* cbK;
    const clo_half* cbV;
    const int32_t* idx;
    const clo_half* pK;
    const clo_half* pV;
    const int32_t* persist_ids;
    int k, C, Np, T, B, Hkv;
    int tp, tc;             // tiles of a persistent / Cache Buffer segment
    long long per_b;        // tiles per batch row

    // Shared scratch: [0] = ids valid flag, [1 .. Hkv] slot -> KV head.
    static size_t smem_ints(int Hkv_, int /*B*/) { return static_cast<size_t>(Hkv_) + 4; }

    __device__ void cta_init(int* sm, int32_t* err_flag, bool report) const {
        if (threadIdx.x == 0) {
            unsigned long long used = 0ull;
            int ok = 1;
            for (int j = 0; j < Np; ++j) {
                const int g = persist_ids[j];
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
    __device__ long long num_tiles(const int*) const { return per_b * B; }
    __device__ int seg_of(long long t, const int*) const {
        const int b = static_cast<int>(t / per_b);
        const long long r = t - per_b * b;
        const long long np_tiles = static_cast<long long>(Np) * tp;
        const int slot = r < np_tiles ? static_cast<int>(r / tp)
                                      : Np + static_cast<int>((r - np_tiles) / tc);
        return b * Hkv + slot;
    }
    __device__ Seg segment(int s, const int* sm) const {
        Seg g;
        g.b = s / Hkv;
        const int slot = s - g.b * Hkv;
        g.kv = sm[1 + slot];
        const bool pers = slot < Np;
        g.slot = pers ? slot : -1;
        g.n_tok = pers ? T : k;
        g.ntiles = pers ? tp : tc;
        g.first = per_b * g.b + (pers ? static_cast<long long>(slot) * tp
                                      : static_cast<long long>(Np) * tp +
                                            static_cast<long long>(slot - Np) * tc);
        return g;
    }
    __device__ bool all_bad(const int* sm) const { return sm[0] == 0; }
    // Row `row` (0..15) of tile `tile_in` of segment g: element offset of the
    // row from the returned base pointers; in_range / ok as described.
    __device__ void row(const Seg& g, int tile_in, int r, const int* sm, const clo_half*& bk,
                        const clo_half*& bv, long long& off, bool& in_range, bool& ok) const {
        const int tok = tile_in * TILE + r;
        in_range = tok < g.n_tok;
        if (g.slot >= 0) {
            bk = pK;
            bv = pV;
            off = (static_cast<long long>(g.b) * Np + g.slot) * T + tok;
            ok = sm[0] != 0;
        } else {
            bk = cbK;
            bv = cbV;
            const long long hb = static_cast<long long>(g.b) * Hkv + g.kv;
            int iv = 0;
            if (in_range) iv = __ldg(idx + hb * k + tok);
            ok = (sm[0] != 0) && iv >= 0 && iv < C;
            off = hb * C + (ok ? iv : 0);
        }
        off *= D;
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
    __device__ Seg segment(int s, const int* sm) const {
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
    __device__ void row(const Seg& g, int tile_in, int r, const int*, const clo_half*& bk,
                        const clo_half*& bv, long long& off, bool& in_range, bool& ok) const {
        bk = kc;
        bv = vc;
        in_range = tile_in * TILE + r < g.n_tok;
        const int blk = __ldg(block_table + static_cast<long long>(g.b) * max_blocks + tile_in);
        ok = blk >= 0 && blk < num_blocks;
        off = ((static_cast<long long>(ok ? blk : 0) * Hkv + g.kv) * TILE + r) * D;
    }
};

// ---------------------------------------------------------------- tile copy
// Issues the cp.async copies of one tile (16 K rows + 16 V rows) into a ring
// stage and records its row masks (bits 0-15 valid rows, 16-31 bad rows).
template <class Geo>
__device__ __forceinline__ void issue_tile(const Geo& geo, const int* gsm, long long t,
                                           uint32_t stage, uint32_t* mask_slot, int lane) {
    const int s = geo.seg_of(t, gsm);
    const Seg sg = geo.segment(s, gsm);
    const int tile_in = static_cast<int>(t - sg.first);
    const clo_half* bk;
    const clo_half* bv;
    long long off;
    bool in_range, ok;
    geo.row(sg, tile_in, lane & 15, gsm, bk, bv, off, in_range, ok);
    const unsigned valid = __ballot_sync(FULL_MASK, in_range && ok) & 0xffffu;
    const unsigned bad = __ballot_sync(FULL_MASK, in_range && !ok) & 0xffffu;
    if (lane == 0) *mask_slot = valid | (bad << 16);
    const int chunk = lane & 15;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = (lane >> 4) + 2 * i;
        const long long ro = __shfl_sync(FULL_MASK, off, r);
        const bool v = (valid >> r) & 1u;
        const uint32_t dst = stage + r * ROW_BYTES + ((chunk ^ (r & 7)) << 4);
        const clo_half* sk = v ? bk + ro + chunk * 8 : bk;
        const clo_half* sv = v ? bv + ro + chunk * 8 : bv;
        cp_async_16(dst, sk, v ? 16 : 0);
        cp_async_16(dst + KV_TILE_BYTES, sv, v ? 16 : 0);
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
    float s[4] = {0.f, 0.f, 0.f, 0.f};
    const int arow = lane & 15;
    const int ahi = lane >> 4;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        uint32_t a[4];
        const int chunk = 2 * kk + ahi;
        ldmatrix_x4(a, Ks + arow * ROW_BYTES + ((chunk ^ (arow & 7)) << 4));
        mma_16816(s, a, qb[kk][0], qb[kk][1]);
    }
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
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        w.acc[i][0] *= al0;
        w.acc[i][1] *= al1;
        w.acc[i][2] *= al0;
        w.acc[i][3] *= al1;
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
    float* m;     // [WARPS][MAXG]
    float* l;     // [WARPS][MAXG]
    int* bad;     // [WARPS]
    float* o;     // [WARPS][G][OSTRIDE]
};

// Combines the warps' states for segment s; writes the final output when the
// whole segment is inside this CTA, else this CTA's partial.
__device__ __forceinline__ void flush_segment(const AttnOut& o, const MergeSmem& ms, WarpState& w,
                                              const Seg& sg, int s, long long c0, long long c1,
                                              bool force_bad, int warp, int lane) {
    float l0 = w.l0, l1 = w.l1;
#pragma unroll
    for (int off = 4; off <= 16; off <<= 1) {
        l0 += __shfl_xor_sync(FULL_MASK, l0, off);
        l1 += __shfl_xor_sync(FULL_MASK, l1, off);
    }
    const int h0 = 2 * (lane & 3), h1 = h0 + 1;
    if (lane < 4) {
        ms.m[warp * MAXG + h0] = w.m0;
        ms.m[warp * MAXG + h1] = w.m1;
        ms.l[warp * MAXG + h0] = l0;
        ms.l[warp * MAXG + h1] = l1;
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
    int bad = force_bad ? 1 : 0;
    for (int x = 0; x < ATTN_WARPS; ++x) bad |= ms.bad[x];
    const bool complete = sg.first >= c0 && sg.first + sg.ntiles <= c1;
    for (int it = threadIdx.x; it < G * D; it += ATTN_THREADS) {
        const int h = it >> 7, dd = it & (D - 1);
        float M = -INFINITY;
        for (int x = 0; x < ATTN_WARPS; ++x) M = fmaxf(M, ms.m[x * MAXG + h]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
            for (int x = 0; x < ATTN_WARPS; ++x) {
                const float mw = ms.m[x * MAXG + h];
                if (mw != -INFINITY) {
                    const float e = fast_exp2(mw - M);
                    L = fmaf(ms.l[x * MAXG + h], e, L);
                    O = fmaf(ms.o[(x * G + h) * OSTRIDE + dd], e, O);
                }
            }
        }
        const bool empty = !(L > 0.f);
        if (complete) {
            const size_t row = static_cast<size_t>(sg.b) * o.Hq + static_cast<size_t>(sg.kv) * G + h;
            const float val = (bad || empty) ? 0.f : O / L;
            o.out[row * D + dd] = __half_as_ushort(__float2half_rn(val));
            if (o.lse != nullptr && dd == 0)
                o.lse[row] = (bad || empty) ? -INFINITY : (M + log2f(L)) * LN2;
        } else {
            const size_t slot = static_cast<size_t>(blockIdx.x) + static_cast<size_t>(s);
            o.ws_o[(slot * G + h) * D + dd] = empty ? 0.f : O / L;
            if (dd == 0) o.ws_lse[slot * G + h] = bad ? INFINITY : (empty ? -INFINITY : M + log2f(L));
        }
    }
    __syncthreads();
}

template <class Geo>
__global__ void __launch_bounds__(ATTN_THREADS, 1)
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
    geo.cta_init(gsm, o.err_flag, blockIdx.x == 0);
    __syncthreads();
    const bool all_bad = geo.all_bad(gsm);

    // The paged tile count is only known on the device: CTAs beyond it retire,
    // so no CTA ever owns an empty range (the merge relies on that).
    const long long N = geo.num_tiles(gsm);
    const int C = static_cast<int>(min(static_cast<long long>(gridDim.x), N));
    if (static_cast<int>(blockIdx.x) >= C) return;
    const long long c0 = N * blockIdx.x / C, c1 = N * (blockIdx.x + 1) / C;
    const int s_first = geo.seg_of(c0, gsm), s_last = geo.seg_of(c1 - 1, gsm);

    const long long my0 = c0 + warp;
    const int nj = my0 < c1 ? static_cast<int>((c1 - my0 + ATTN_WARPS - 1) / ATTN_WARPS) : 0;
    const uint32_t ring = smem_u32(smem) + warp * ATTN_STAGES * STAGE_BYTES;
    uint32_t* my_masks = masks + warp * ATTN_STAGES;

#pragma unroll
    for (int j = 0; j < ATTN_STAGES - 1; ++j) {
        if (j < nj)
            issue_tile(geo, gsm, my0 + static_cast<long long>(j) * ATTN_WARPS,
                       ring + j * STAGE_BYTES, my_masks + j, lane);
        cp_async_commit();
    }

    int jc = 0;
    WarpState w;
    for (int s = s_first; s <= s_last; ++s) {
        const Seg sg = geo.segment(s, gsm);
        if (sg.ntiles == 0) continue;  // empty requests are written before the launch loop
        const long long seg_end = sg.first + sg.ntiles;
        uint32_t qb[8][2];
        load_q(o, sg, lane, qb);
        state_reset(w);
        while (jc < nj) {
            const long long t = my0 + static_cast<long long>(jc) * ATTN_WARPS;
            if (t >= seg_end) break;
            cp_async_wait<ATTN_STAGES - 2>();
            __syncwarp();
            const int jn = jc + ATTN_STAGES - 1;
            if (jn < nj)
                issue_tile(geo, gsm, my0 + static_cast<long long>(jn) * ATTN_WARPS,
                           ring + (jn % ATTN_STAGES) * STAGE_BYTES, my_masks + jn % ATTN_STAGES,
                           lane);
            cp_async_commit();
            const int st = jc % ATTN_STAGES;
            const uint32_t mw = *reinterpret_cast<volatile uint32_t*>(my_masks + st);
            w.bad |= static_cast<int>(mw >> 16);
            compute_tile(ring + st * STAGE_BYTES, mw & 0xffffu, qb, o.scale_log2, w, lane);
            ++jc;
        }
        flush_segment(o, ms, w, sg, s, c0, c1, all_bad, warp, lane);
    }
    cp_async_wait<0>();
}

// Zeroes the outputs of requests with no tokens (paged only).
__global__ void paged_zero_empty_kernel(const int32_t* __restrict__ ctx_len, int B, int max_tok,
                                        int Hq, clo_half* __restrict__ out, float* __restrict__ lse) {
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

// Merges the per-CTA partials of every segment cut by a CTA boundary.  Block
// i looks at the boundary between CTA i and i+1 and handles the segment that
// straddles it if that segment starts inside CTA i (so each cut segment is
// merged exactly once).
template <class Geo>
__global__ void __launch_bounds__(MERGE_THREADS)
    attn_merge_kernel(const Geo geo, const AttnOut o, int C) {
    extern __shared__ __align__(16) uint8_t msmem[];
    const int G = o.G;
    const int items = G * 32;             // (head, 4-float column)
    const int ngrp = MERGE_THREADS / items;
    float* Mg = reinterpret_cast<float*>(msmem);        // [ngrp][G]
    float* Lg = Mg + ngrp * MAXG;                       // [ngrp][G]
    int* Bg = reinterpret_cast<int*>(Lg + ngrp * MAXG); // [ngrp][G]
    float4* Og = reinterpret_cast<float4*>(Bg + ngrp * MAXG);  // [ngrp][G][32]
    int* gsm = reinterpret_cast<int*>(Og + ngrp * items);

    geo.cta_init(gsm, nullptr, false);
    __syncthreads();
    const long long N = geo.num_tiles(gsm);
    const int Ce = static_cast<int>(min(static_cast<long long>(C), N));  // CTAs that had work
    const int i = blockIdx.x;
    if (i >= Ce - 1) return;
    const long long start_i = N * i / Ce, tb = N * (i + 1) / Ce;
    const int s = geo.seg_of(tb, gsm);
    const Seg sg = geo.segment(s, gsm);
    if (!(sg.first < tb && sg.first >= start_i)) return;
    const long long last = sg.first + sg.ntiles - 1;
    const int c_hi = static_cast<int>(((last + 1) * Ce - 1) / N);
    const int P = c_hi - i + 1;

    const int it = threadIdx.x % items, grp = threadIdx.x / items;
    const int h = it >> 5, col = it & 31;
    if (grp < ngrp) {
        float M = -INFINITY;
        int bad = 0;
        for (int p = grp; p < P; p += ngrp) {
            const float x = o.ws_lse[(static_cast<size_t>(i + p) + s) * G + h];
            if (x == INFINITY) bad = 1;
            else M = fmaxf(M, x);
        }
        float L = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (M != -INFINITY) {
            for (int p = grp; p < P; p += ngrp) {
                const size_t slot = static_cast<size_t>(i + p) + s;
                const float x = o.ws_lse[slot * G + h];
                if (x == INFINITY || x == -INFINITY) continue;
                const float e = fast_exp2(x - M);
                const float4 v = reinterpret_cast<const float4*>(o.ws_o + (slot * G + h) * D)[col];
                L += e;
                acc.x = fmaf(v.x, e, acc.x);
                acc.y = fmaf(v.y, e, acc.y);
                acc.z = fmaf(v.z, e, acc.z);
                acc.w = fmaf(v.w, e, acc.w);
            }
        }
        if (col == 0) {
            Mg[grp * MAXG + h] = M;
            Lg[grp * MAXG + h] = L;
            Bg[grp * MAXG + h] = bad;
        }
        Og[grp * items + it] = acc;
    }
    __syncthreads();
    if (grp == 0) {
        float M = -INFINITY;
        int bad = 0;
        for (int g2 = 0; g2 < ngrp; ++g2) {
            M = fmaxf(M, Mg[g2 * MAXG + h]);
            bad |= Bg[g2 * MAXG + h];
        }
        float L = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (M != -INFINITY) {
            for (int g2 = 0; g2 < ngrp; ++g2) {
                const float mg = Mg[g2 * MAXG + h];
                if (mg == -INFINITY) continue;
                const float e = fast_exp2(mg - M);
                const float4 v = Og[g2 * items + it];
                L = fmaf(Lg[g2 * MAXG + h], e, L);
                acc.x = fmaf(v.x, e, acc.x);
                acc.y = fmaf(v.y, e, acc.y);
                acc.z = fmaf(v.z, e, acc.z);
                acc.w = fmaf(v.w, e, acc.w);
            }
        }
        const bool empty = !(L > 0.f);
        const size_t row = static_cast<size_t>(sg.b) * o.Hq + static_cast<size_t>(sg.kv) * G + h;
        const float inv = (bad || empty) ? 0.f : 1.f / L;
        __half2 lo = __floats2half2_rn(acc.x * inv, acc.y * inv);
        __half2 hi = __floats2half2_rn(acc.z * inv, acc.w * inv);
        uint2 pk;
        pk.x = *reinterpret_cast<uint32_t*>(&lo);
        pk.y = *reinterpret_cast<uint32_t*>(&hi);
        reinterpret_cast<uint2*>(o.out + row * D)[col] = pk;
        if (o.lse != nullptr && col == 0)
            o.lse[row] = (bad || empty) ? -INFINITY : (M + log2f(L)) * LN2;
    }
}

// ---------------------------------------------------------------- host side

static int device_sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev] = n;
    }
    return cache[dev];
}

static bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Raises a kernel's dynamic shared-memory limit once per (kernel, device).
static bool smem_attr_set(const void* func, int bytes) {
    static std::mutex mu;
    static const void* done_func[64];
    static int done_dev[64];
    static int n_done = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n_done; ++i)
        if (done_func[i] == func && done_dev[i] == dev) return true;
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
        cudaSuccess)
        return false;
    if (n_done < 64) {
        done_func[n_done] = func;
        done_dev[n_done] = dev;
        ++n_done;
    }
    return true;
}

static size_t partial_bytes(long long slots, int G) {
    const size_t o = static_cast<size_t>(slots) * G * D * sizeof(float);
    const size_t l = static_cast<size_t>(slots) * G * sizeof(float);
    return ((o + 255) / 256) * 256 + ((l + 255) / 256) * 256;
}

static size_t workspace_bytes(int B, int Hq, int Hkv, int d, int num_ctas) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d != D || num_ctas < 0) return 0;
    const int G = Hq / Hkv;
    if (G > MAXG) return 0;
    int C = num_ctas > 0 ? num_ctas : device_sm_count();
    if (C <= 0) return 0;
    return partial_bytes(static_cast<long long>(C) + static_cast<long long>(B) * Hkv, G);
}

static size_t attn_smem_bytes(int G, size_t geo_ints) {
    return static_cast<size_t>(ATTN_WARPS) * ATTN_STAGES * STAGE_BYTES +
           ATTN_WARPS * ATTN_STAGES * sizeof(uint32_t) + 2 * ATTN_WARPS * MAXG * sizeof(float) +
           ATTN_WARPS * sizeof(int) + static_cast<size_t>(ATTN_WARPS) * G * OSTRIDE * sizeof(float) +
           geo_ints * sizeof(int);
}

static size_t merge_smem_bytes(int G, size_t geo_ints) {
    const int items = G * 32;
    const int ngrp = MERGE_THREADS / items;
    return static_cast<size_t>(ngrp) * MAXG * 3 * sizeof(float) +
           static_cast<size_t>(ngrp) * items * sizeof(float4) + geo_ints * sizeof(int);
}

template <class Geo>
static clo_status launch_attention(const Geo& geo, AttnOut o, long long n_tiles_host_bound,
                                   size_t geo_ints, int S, void* workspace, size_t ws_bytes,
                                   const clo_attn_opts* opts, cudaStream_t stream) {
    if (!smem_attr_set(reinterpret_cast<const void*>(attn_split_kernel<Geo>), SMEM_LIMIT))
        return CLO_ERR_CUDA;
    const size_t smem = attn_smem_bytes(o.G, geo_ints);
    const size_t msmem = merge_smem_bytes(o.G, geo_ints);
    if (smem > static_cast<size_t>(SMEM_LIMIT) || msmem > 48 * 1024) return CLO_ERR_UNSUPPORTED;

    int C = (opts != nullptr && opts->num_ctas > 0) ? opts->num_ctas : device_sm_count();
    if (C <= 0) return CLO_ERR_CUDA;
    // Never more CTAs than tiles (no CTA gets an empty range) and at least one
    // tile per warp where the problem allows.
    const long long cap = n_tiles_host_bound / ATTN_WARPS;
    if (C > cap) C = static_cast<int>(cap > 0 ? cap : 1);
    if (C > n_tiles_host_bound) C = static_cast<int>(n_tiles_host_bound);
    if (C < 1) C = 1;
    const size_t need = partial_bytes(static_cast<long long>(C) + S, o.G);
    if (workspace == nullptr || ws_bytes < need || !aligned(workspace, 16)) return CLO_ERR_WORKSPACE;
    const long long slots = static_cast<long long>(C) + S;
    o.ws_o = static_cast<float*>(workspace);
    o.ws_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                        ((static_cast<size_t>(slots) * o.G * D * sizeof(float) + 255) / 256) * 256);

    // External records so that, under stream capture, they become event nodes
    // of the graph (re-recorded on every replay).
    if (opts != nullptr && opts->ev_begin != nullptr &&
        cudaEventRecordWithFlags(opts->ev_begin, stream, cudaEventRecordExternal) != cudaSuccess)
        return CLO_ERR_CUDA;
    attn_split_kernel<Geo><<<C, ATTN_THREADS, smem, stream>>>(geo, o);
    if (cudaGetLastError() != cudaSuccess) return CLO_ERR_CUDA;
    if (opts != nullptr && opts->ev_end != nullptr &&
        cudaEventRecordWithFlags(opts->ev_end, stream, cudaEventRecordExternal) != cudaSuccess)
        return CLO_ERR_CUDA;
    if (C >= 2) {
        attn_merge_kernel<Geo><<<C - 1, MERGE_THREADS, msmem, stream>>>(geo, o, C);
        if (cudaGetLastError() != cudaSuccess) return CLO_ERR_CUDA;
    }
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

extern "C" clo_status clo_hybrid_decode_attn(const clo_half* q, const clo_half* cbK,
                                             const clo_half* cbV, const int32_t* idx, int k, int C,
                                             const clo_half* pK, const clo_half* pV,
                                             const int32_t* persist_ids, int Np, int T, int B,
                                             int Hq, int Hkv, int d, float scale, clo_half* out,
                                             float* lse, void* workspace, size_t ws_bytes,
                                             int32_t* err_flag, const clo_attn_opts* opts,
                                             cudaStream_t stream) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || Np < 0 || Np > Hkv)
        return CLO_ERR_INVALID_ARG;
    if (B == 0) return CLO_OK;  // empty batch: nothing to compute
    if (q == nullptr || out == nullptr) return CLO_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !isfinite(scale)) return CLO_ERR_INVALID_ARG;
    const int G = Hq / Hkv;
    if (d != D || G > MAXG || Hkv > MAX_HKV_HYBRID) return CLO_ERR_UNSUPPORTED;
    const bool has_cb = Np < Hkv;
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
    geo.per_b = static_cast<long long>(Np) * (Np > 0 ? geo.tp : 0) +
                static_cast<long long>(Hkv - Np) * (has_cb ? geo.tc : 0);
    const long long N = geo.per_b * B;

    AttnOut o{};
    o.q = q;
    o.out = out;
    o.lse = lse;
    o.err_flag = err_flag;
    o.scale_log2 = scale * LOG2E;
    o.Hq = Hq;
    o.G = G;
    return launch_attention(geo, o, N, HybridGeo::smem_ints(Hkv, B), B * Hkv, workspace,
                            ws_bytes, opts, stream);
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
    paged_zero_empty_kernel<<<B, 128, 0, stream>>>(ctx_len, B, max_blocks * TILE, Hq, out, lse);
    if (cudaGetLastError() != cudaSuccess) return CLO_ERR_CUDA;
    // The tile count depends on device-resident lengths; size the grid for the
    // largest possible stream (CTAs never exceed the true count, see kernel).
    const long long bound = static_cast<long long>(B) * Hkv * max_blocks;
    return launch_attention(geo, o, bound, PagedGeo::smem_ints(Hkv, B), B * Hkv, workspace,
                            ws_bytes, opts, stream);
}
