// Expert contractions of a block: every selected expert's SwiGLU MLP on the
// rows routed to it, the shared experts on every row, and the stand-alone Q8_0
// block matmul, all through one persistent kernel.
//
// Pages: "Run Kimi 3.1 locally on one GPU": MXFP4 experts, one file per expert
// (section "One GPU, three storage tiers"); a block reads each expert once for
// all its rows, and its rows run the same arithmetic as plain steps (section
// "A drafter that leaves the answer unchanged").  The spine (here: the shared
// experts) is Q8_0 and its matmuls load each weight once for all rows.
//
// Design (GB300):
// * One CTA per SM, 8 consumer warps + 1 producer warp.  The producer claims
//   work items from a global counter in order, and streams each item's weight
//   tiles HBM -> shared memory with TMA (3-D tensor maps over the slab pool,
//   128-byte swizzle) into an 8-stage mbarrier ring.  Every weight byte of a
//   block is read from HBM exactly once.
// * Work items: gate/up items (16 output rows of both matrices, full K) and
//   down items (64 output rows, full K).  Items are ordered gate/up of expert
//   v, then down of expert v-2, so a down item rarely waits; it waits (bounded)
//   on a per-expert counter of finished gate/up items.
// * Consumers convert E2M1 codes to f16 with cvt.rn.f16x2.e2m1x2 (exact) and
//   int8 with a mantissa trick (exact), and multiply with warp-level tensor-core
//   MMAs (m16n8k16, fp32 accumulate) against the block's rows: x pre-scaled to
//   f16 by a power of two, h split into f16 hi + lo parts.  Each K group of 32
//   forms its own MMA partial, which is then scaled by that group's E8M0 or
//   fp16 scale, so the weights enter exactly.
// * A row's arithmetic never depends on the other rows of the block: K is
//   always reduced in the same order, the row's tensor-core column does not
//   change its result, and scale exponents are per row.
#include <algorithm>
#include <mutex>

#include "common.cuh"

namespace moe {

constexpr int EX_CW = 8;                      // consumer warps
constexpr int EX_CT = EX_CW * 32;             // consumer threads
constexpr int EX_THREADS = EX_CT + 32;        // + producer warp
// ring stages: the consumers, not the copies, set the pace (~15 GB/s per SM), so a
// deeper ring only adds bytes in flight, which lengthens the memory round trips of
// the kernels running beside it (the routing)
constexpr int EX_NST = 4;
constexpr int EX_CTAS_PER_SM = 1;
constexpr int EX_CODE_BYTES = 16384;
constexpr int EX_STAGE = 17408;               // codes + scales
constexpr int EX_NT = 2;                      // n-tiles of 8 rows: up to 16 rows per expert
constexpr int EX_RED_FLOATS = EX_CW * 4 * EX_NT * 4 * 32;  // one down-item reduction
constexpr int EX_RED_GU = EX_CW * 2 * EX_NT * 4 * 32;      // a gate/up item uses half of it
constexpr int EX_XS_BYTES = 57344;             // the block's f16 rows, kept in shared memory when they fit
constexpr size_t EX_SMEM = (size_t)EX_NST * EX_STAGE + EX_RED_FLOATS * 4 + EX_XS_BYTES + 64 + 1024 + 1024;

enum { IT_GU = 0, IT_DN = 1 };
enum { J_LAYER = 0, J_Q8_SWIGLU = 1, J_Q8_PLAIN = 2 };

struct Geom {
    int row_bytes, bi, cb, nbox, sb, flat, chunks, gps, rows_item;
    int fast;    // full-width swizzled stages: the unrolled per-warp tile paths apply
    int merged;  // the maps were built by pool_maps for such stages: a stage is one TMA
                 // box of codes (gate and up together) plus one of scales
    uint32_t tx;
};

struct ExParams {
    CUtensorMap map[12];  // routed then shared: gate codes, gate scales, up codes, up scales, down codes, down scales
    Geom geom[4];         // routed gate/up, routed down, shared gate/up, shared down
    int job, fmt_routed, fmt_shared;
    int k_gu, m_gu, k_dn, m_dn;
    int top_k, n_rows, n_shared;
    int n_gu, n_dn, lag;
    int debug_gu, accum;
    int routed_off;  // layer job without the routed experts (they run on the block-scaled path)
    int work_word, exit_word;  // ctrl words of this launch's work counter and exit counter
    // shared-expert launch: the block's bf16 rows, turned into the f16 copy (x16, xexp)
    // by the first CTAs to start; null when x16 was written by an earlier kernel
    const uint16_t* x_rows;
    int dep_at_end;  // wait for the previous kernel on the stream at the end, not the start
    int x_smem;      // with x_rows: every CTA keeps its own f16 copy in shared memory (N d <= EX_XS_BYTES / 2)
    const int* expert_slot;
    const uint32_t* slot_ready;
    int n_slots;
    uint32_t* ctrl;
    const int* uexp;
    const int* uorder;   // MOE_MODE_ORDERED: position -> index into uexp/off, else null
    const int* off;
    const int* pair;
    const __half* x16;
    const int* xexp;
    uint32_t* gu_done;
    uint32_t* hmax;
    float* h;
    float* dbg_g;
    float* dbg_u;
    float* out_shared;
    float* y_part;
    int64_t pairs_cap;
    // plain Q8_0 job: each 64-row down item is split into ksplit K ranges (0 or 1: not
    // split); the ranges' sums go to kpart [ksplit][n_rows][m_dn] and the last of a row
    // block's items to finish (karrive [m_dn / 64]) adds them in range order
    int ksplit;
    float* kpart;
    uint32_t* karrive;
};

struct Meta {
    int item, type, v, blk, chunk, nchunks, slot;
    int c0;  // first chunk of the item (its chunks are c0 .. nchunks - 1)
};

__device__ __forceinline__ int ksplit_of(const ExParams& p) { return p.ksplit > 1 ? p.ksplit : 1; }

__device__ __forceinline__ void item_counts(const ExParams& p, bool& has_gu, bool& has_dn, int& lag) {
    has_gu = p.job != J_Q8_PLAIN;
    has_dn = p.job != J_Q8_SWIGLU;
    lag = (has_gu && has_dn) ? p.lag : 0;
}

__device__ __forceinline__ int total_items(const ExParams& p, int V) {
    bool g, d;
    int lag;
    item_counts(p, g, d, lag);
    return V * ((g ? p.n_gu : 0) + (d ? p.n_dn * ksplit_of(p) : 0));
}

// Item order: round i holds the gate/up items of expert i, then the down items
// of expert i - lag.
__device__ void decode_item(const ExParams& p, int V, int item, int& type, int& v, int& blk) {
    bool has_gu, has_dn;
    int lag;
    item_counts(p, has_gu, has_dn, lag);
    int rest = item;
    for (int i = 0; i < V + lag; i++) {
        if (has_gu && i < V) {
            if (rest < p.n_gu) {
                type = IT_GU;
                v = i;
                blk = rest;
                return;
            }
            rest -= p.n_gu;
        }
        const int vd = i - lag;
        if (has_dn && vd >= 0 && vd < V) {
            // a split down item's blk is row block * ksplit + K range
            const int n_dn = p.n_dn * ksplit_of(p);
            if (rest < n_dn) {
                type = IT_DN;
                v = vd;
                blk = rest;
                return;
            }
            rest -= n_dn;
        }
    }
    type = IT_GU;
    v = 0;
    blk = 0;
}

// shared-memory address of the code bytes at byte offset `ob` of row `row`
// inside a matrix region of `rows` rows laid out as TMA boxes of `bi` bytes.
__device__ __forceinline__ uint32_t code_addr(uint32_t base, const Geom& g, int rows, int row, int ob) {
    const int box = ob / g.bi;
    const int in = ob - box * g.bi;
    const int swm = (g.bi == 128) ? 7 : 0;
    return base + (uint32_t)(box * g.bi * rows + row * g.bi + ((((in >> 4) ^ (row & swm)) << 4) | (in & 15)));
}

// A-fragment words of rows r0 (= lane/4) and r1 (= r0+8) for this thread's 8
// K values of group q: four f16x2 for the first MMA of the group, four for the second.
template <int FMT>
__device__ __forceinline__ void load_a(uint32_t cbase, const Geom& g, int rows, int r0, int r1, int q, int i,
                                       uint32_t (&a0)[4], uint32_t (&a1)[4]) {
    if (FMT == MOE_FMT_MXFP4) {
        const int ob = 16 * q + 4 * i;
        const uint32_t w0 = lds32(code_addr(cbase, g, rows, r0, ob));
        const uint32_t w1 = lds32(code_addr(cbase, g, rows, r1, ob));
        uint32_t x0, x1, x2, x3, y0, y1, y2, y3;
        e2m1x8_to_f16x2(w0, x0, x1, x2, x3);
        e2m1x8_to_f16x2(w1, y0, y1, y2, y3);
        a0[0] = x0; a0[1] = y0; a0[2] = x1; a0[3] = y1;
        a1[0] = x2; a1[1] = y2; a1[2] = x3; a1[3] = y3;
    } else {
        const int ob = 32 * q + 8 * i;
        const uint2 w0 = lds64(code_addr(cbase, g, rows, r0, ob));
        const uint2 w1 = lds64(code_addr(cbase, g, rows, r1, ob));
        uint32_t x0, x1, x2, x3, y0, y1, y2, y3;
        s8x4_to_f16x2(w0.x, x0, x1);
        s8x4_to_f16x2(w0.y, x2, x3);
        s8x4_to_f16x2(w1.x, y0, y1);
        s8x4_to_f16x2(w1.y, y2, y3);
        a0[0] = x0; a0[1] = y0; a0[2] = x1; a0[3] = y1;
        a1[0] = x2; a1[1] = y2; a1[2] = x3; a1[3] = y3;
    }
}

template <int FMT>
__device__ __forceinline__ float load_scale(uint32_t sbase, const Geom& g, int row, int q) {
    if (FMT == MOE_FMT_MXFP4) return e8m0_to_f32(lds8(sbase + row * g.sb + q));
    return __half2float(__ushort_as_half((unsigned short)lds16(sbase + row * g.sb + 2 * q)));
}

__device__ __forceinline__ void fma4(float (&acc)[4], float s0, float s1, const float (&pp)[4]) {
    acc[0] = fmaf(s0, pp[0], acc[0]);
    acc[1] = fmaf(s0, pp[1], acc[1]);
    acc[2] = fmaf(s1, pp[2], acc[2]);
    acc[3] = fmaf(s1, pp[3], acc[3]);
}

// one stage of a gate/up item
template <int FMT>
__device__ __forceinline__ void gu_stage(uint32_t st, const Geom& g, int chunk, int cw, int lane, int NT,
                                         const __half* const (&xrow)[EX_NT], const bool (&bval)[EX_NT],
                                         float (&ag)[EX_NT][4], float (&au)[EX_NT][4]) {
    const int gq = lane >> 2, i = lane & 3;
    const uint32_t gateC = st, upC = st + g.nbox * g.bi * 16;
    const uint32_t gateS = st + EX_CODE_BYTES, upS = st + EX_CODE_BYTES + 512;
    for (int q = cw; q < g.gps; q += EX_CW) {
        const int kk = (chunk * g.gps + q) * 32 + 8 * i;
        uint4 bx[EX_NT];
#pragma unroll
        for (int nt = 0; nt < EX_NT; nt++) {
            bx[nt] = make_uint4(0, 0, 0, 0);
            if (nt < NT && bval[nt]) bx[nt] = *reinterpret_cast<const uint4*>(xrow[nt] + kk);
        }
        uint32_t g0[4], g1[4], u0[4], u1[4];
        load_a<FMT>(gateC, g, 16, gq, gq + 8, q, i, g0, g1);
        load_a<FMT>(upC, g, 16, gq, gq + 8, q, i, u0, u1);
        const float sg0 = load_scale<FMT>(gateS, g, gq, q), sg1 = load_scale<FMT>(gateS, g, gq + 8, q);
        const float su0 = load_scale<FMT>(upS, g, gq, q), su1 = load_scale<FMT>(upS, g, gq + 8, q);
#pragma unroll
        for (int nt = 0; nt < EX_NT; nt++) {
            if (nt < NT) {
                float pg[4] = {0.f, 0.f, 0.f, 0.f}, pu[4] = {0.f, 0.f, 0.f, 0.f};
                mma_f16(pg, g0[0], g0[1], g0[2], g0[3], bx[nt].x, bx[nt].y);
                mma_f16(pg, g1[0], g1[1], g1[2], g1[3], bx[nt].z, bx[nt].w);
                mma_f16(pu, u0[0], u0[1], u0[2], u0[3], bx[nt].x, bx[nt].y);
                mma_f16(pu, u1[0], u1[1], u1[2], u1[3], bx[nt].z, bx[nt].w);
                fma4(ag[nt], sg0, sg1, pg);
                fma4(au[nt], su0, su1, pu);
            }
        }
    }
}

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// one stage of a down item (4 M-tiles of 16 rows)
template <int FMT>
__device__ __forceinline__ void dn_stage(uint32_t st, const Geom& g, int chunk, int cw, int lane, int NT,
                                         const float* const (&hrow)[EX_NT], const float (&hs)[EX_NT],
                                         const bool (&bval)[EX_NT], float (&acc)[4][EX_NT][4]) {
    const int gq = lane >> 2, i = lane & 3;
    const uint32_t C = st, S = st + EX_CODE_BYTES;
    for (int q = cw; q < g.gps; q += EX_CW) {
        const int kk = (chunk * g.gps + q) * 32 + 8 * i;
        uint32_t hi[EX_NT][4], lo[EX_NT][4];
#pragma unroll
        for (int nt = 0; nt < EX_NT; nt++) {
#pragma unroll
            for (int t = 0; t < 4; t++) hi[nt][t] = lo[nt][t] = 0u;
            if (nt < NT && bval[nt]) {
                const float4 va = __ldca(reinterpret_cast<const float4*>(hrow[nt] + kk));
                const float4 vb = __ldca(reinterpret_cast<const float4*>(hrow[nt] + kk + 4));
                const float v[8] = {va.x * hs[nt], va.y * hs[nt], va.z * hs[nt], va.w * hs[nt],
                                    vb.x * hs[nt], vb.y * hs[nt], vb.z * hs[nt], vb.w * hs[nt]};
#pragma unroll
                for (int t = 0; t < 4; t++) {
                    const __half2 hh = __floats2half2_rn(v[2 * t], v[2 * t + 1]);
                    const float2 back = __half22float2(hh);
                    hi[nt][t] = *reinterpret_cast<const uint32_t*>(&hh);
                    lo[nt][t] = pack_h2(v[2 * t] - back.x, v[2 * t + 1] - back.y);
                }
            }
        }
#pragma unroll
        for (int mt = 0; mt < 4; mt++) {
            const int r0 = mt * 16 + gq, r1 = r0 + 8;
            uint32_t a0[4], a1[4];
            load_a<FMT>(C, g, 64, r0, r1, q, i, a0, a1);
            const float s0 = load_scale<FMT>(S, g, r0, q), s1 = load_scale<FMT>(S, g, r1, q);
#pragma unroll
            for (int nt = 0; nt < EX_NT; nt++) {
                if (nt < NT) {
                    float pp[4] = {0.f, 0.f, 0.f, 0.f};
                    mma_f16(pp, a0[0], a0[1], a0[2], a0[3], hi[nt][0], hi[nt][1]);
                    mma_f16(pp, a1[0], a1[1], a1[2], a1[3], hi[nt][2], hi[nt][3]);
                    mma_f16(pp, a0[0], a0[1], a0[2], a0[3], lo[nt][0], lo[nt][1]);
                    mma_f16(pp, a1[0], a1[1], a1[2], a1[3], lo[nt][2], lo[nt][3]);
                    fma4(acc[mt][nt], s0, s1, pp);
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Fast paths for full-width stages (128-byte swizzled boxes, 512 code bytes per
// row per gate/up stage, 256 per down stage).  Warp w owns the T consecutive
// scale groups q = w*T + t of every stage, so each thread's shared-memory
// offsets are constants of the kernel and every loop is unrolled.
// ---------------------------------------------------------------------------

template <int FMT>
struct Tiles {
    static constexpr int T_GU = FMT == MOE_FMT_MXFP4 ? 4 : 2;  // groups per warp per gate/up stage
    static constexpr int T_DN = FMT == MOE_FMT_MXFP4 ? 2 : 1;  // groups per warp per down stage
};

// offset of row (lane/4) of the thread's A words for each of its T groups,
// inside a matrix region of R rows made of 128-byte swizzled boxes
template <int FMT, int T, int R>
__device__ __forceinline__ void fast_offsets(int cw, int lane, uint32_t (&aoff)[T]) {
    const int g = lane >> 2, i = lane & 3;
#pragma unroll
    for (int t = 0; t < T; t++) {
        const int q = cw * T + t;
        int box, chunk, inner;
        if (FMT == MOE_FMT_MXFP4) {
            box = q >> 3;
            chunk = q & 7;
            inner = 4 * i;
        } else {
            box = q >> 2;
            chunk = 2 * (q & 3) + (i >> 1);
            inner = 8 * (i & 1);
        }
        aoff[t] = (uint32_t)(box * 128 * R + g * 128 + ((chunk ^ g) << 4) + inner);
    }
}

// A fragments of rows g (at addr) and g+8 (addr + 1024): same swizzle phase
template <int FMT>
__device__ __forceinline__ void load_a_fast(uint32_t addr, uint32_t (&a0)[4], uint32_t (&a1)[4]) {
    uint32_t x0, x1, x2, x3, y0, y1, y2, y3;
    if (FMT == MOE_FMT_MXFP4) {
        const uint32_t w0 = lds32(addr), w1 = lds32(addr + 1024);
        e2m1x8_to_f16x2(w0, x0, x1, x2, x3);
        e2m1x8_to_f16x2(w1, y0, y1, y2, y3);
    } else {
        const uint2 w0 = lds64(addr), w1 = lds64(addr + 1024);
        s8x4_to_f16x2(w0.x, x0, x1);
        s8x4_to_f16x2(w0.y, x2, x3);
        s8x4_to_f16x2(w1.x, y0, y1);
        s8x4_to_f16x2(w1.y, y2, y3);
    }
    a0[0] = x0; a0[1] = y0; a0[2] = x1; a0[3] = y1;
    a1[0] = x2; a1[1] = y2; a1[2] = x3; a1[3] = y3;
}

// scale t of a word holding the thread's consecutive group scales.  E8M0
// exponents 1..254 are exact powers of two; 0 reads as 0 and 255 as +inf.
template <int FMT>
__device__ __forceinline__ float scale_t(uint32_t w, int t) {
    if (FMT == MOE_FMT_MXFP4) return __uint_as_float(((w >> (8 * t)) & 0xFFu) << 23);
    return __half2float(__ushort_as_half((unsigned short)(w >> (16 * t))));
}

template <int FMT, int T, int NT>
__device__ __forceinline__ void gu_stage_fast(uint32_t st, int chunk, int nchunks, int cw, int lane, bool xg,
                                              const __half* const (&xrow)[EX_NT],
                                              const bool (&bval)[EX_NT], float (&ag)[EX_NT][4],
                                              float (&au)[EX_NT][4]) {
    constexpr int GPS = 8 * T;
    constexpr int SB = FMT == MOE_FMT_MXFP4 ? GPS : 2 * GPS;
    const int gq = lane >> 2, i = lane & 3;
    uint32_t aoff[T];
    fast_offsets<FMT, T, 16>(cw, lane, aoff);
    const uint32_t upC = st + 512 * 16;
    const uint32_t gateS = st + EX_CODE_BYTES + gq * SB + 4 * cw, upS = gateS + 512;
    if (xg && chunk + 1 < nchunks) {
        // the item's next stage reads the next K slice of the same rows (in global
        // memory): T*64 bytes per row and warp, fetched into L1 one 128-byte line per lane i
        constexpr int LINES = (T * 64 + 127) / 128;
#pragma unroll
        for (int nt = 0; nt < NT; nt++)
            if (bval[nt] && i < LINES)
                asm volatile("prefetch.global.L1 [%0];" ::"l"(xrow[nt] + ((chunk + 1) * GPS + cw * T) * 32 + 64 * i));
    }
    const uint32_t sg0 = lds32(gateS), sg1 = lds32(gateS + 8 * SB);
    const uint32_t su0 = lds32(upS), su1 = lds32(upS + 8 * SB);
#pragma unroll
    for (int t = 0; t < T; t++) {
        uint4 bx[NT];
#pragma unroll
        for (int nt = 0; nt < NT; nt++) {
            bx[nt] = make_uint4(0, 0, 0, 0);
            if (bval[nt])
                bx[nt] = *reinterpret_cast<const uint4*>(xrow[nt] + (chunk * GPS + cw * T + t) * 32 + 8 * i);
        }
        uint32_t g0[4], g1[4], u0[4], u1[4];
        load_a_fast<FMT>(st + aoff[t], g0, g1);
        load_a_fast<FMT>(upC + aoff[t], u0, u1);
        const float fg0 = scale_t<FMT>(sg0, t), fg1 = scale_t<FMT>(sg1, t);
        const float fu0 = scale_t<FMT>(su0, t), fu1 = scale_t<FMT>(su1, t);
#pragma unroll
        for (int nt = 0; nt < NT; nt++) {
            {
                float pg[4] = {0.f, 0.f, 0.f, 0.f}, pu[4] = {0.f, 0.f, 0.f, 0.f};
                mma_f16(pg, g0[0], g0[1], g0[2], g0[3], bx[nt].x, bx[nt].y);
                mma_f16(pg, g1[0], g1[1], g1[2], g1[3], bx[nt].z, bx[nt].w);
                mma_f16(pu, u0[0], u0[1], u0[2], u0[3], bx[nt].x, bx[nt].y);
                mma_f16(pu, u1[0], u1[1], u1[2], u1[3], bx[nt].z, bx[nt].w);
                fma4(ag[nt], fg0, fg1, pg);
                fma4(au[nt], fu0, fu1, pu);
            }
        }
    }
}

template <int FMT, int T, int NT>
__device__ __forceinline__ void dn_stage_fast(uint32_t st, int chunk, int nchunks, int cw, int lane,
                                              const float* const (&hrow)[EX_NT],
                                              const float (&hs)[EX_NT], const bool (&bval)[EX_NT],
                                              float (&acc)[4][EX_NT][4]) {
    constexpr int GPS = 8 * T;
    constexpr int SB = FMT == MOE_FMT_MXFP4 ? GPS : 2 * GPS;
    const int gq = lane >> 2, i = lane & 3;
    if (chunk + 1 < nchunks) {
        // the next stage's h values of the same rows: T*128 bytes per row and warp,
        // into L1 one line per lane i < T
#pragma unroll
        for (int nt = 0; nt < NT; nt++)
            if (bval[nt] && i < T)
                asm volatile("prefetch.global.L1 [%0];" ::"l"(hrow[nt] + ((chunk + 1) * GPS + cw * T + i) * 32));
    }
    uint32_t aoff[T];
    fast_offsets<FMT, T, 64>(cw, lane, aoff);
    const uint32_t S = st + EX_CODE_BYTES + gq * SB + 2 * cw;
    uint32_t sw0[4], sw1[4];
#pragma unroll
    for (int mt = 0; mt < 4; mt++) {
        sw0[mt] = lds16(S + mt * 16 * SB);
        sw1[mt] = lds16(S + (mt * 16 + 8) * SB);
    }
#pragma unroll
    for (int t = 0; t < T; t++) {
        uint32_t hi[NT][4], lo[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; nt++) {
            float4 va = make_float4(0.f, 0.f, 0.f, 0.f), vb = va;
            if (bval[nt]) {
                const float* src = hrow[nt] + (chunk * GPS + cw * T + t) * 32 + 8 * i;
                va = __ldca(reinterpret_cast<const float4*>(src));
                vb = __ldca(reinterpret_cast<const float4*>(src + 4));
            }
            const float v[8] = {va.x * hs[nt], va.y * hs[nt], va.z * hs[nt],
                                va.w * hs[nt], vb.x * hs[nt], vb.y * hs[nt],
                                vb.z * hs[nt], vb.w * hs[nt]};
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const __half2 hh = __floats2half2_rn(v[2 * e], v[2 * e + 1]);
                const float2 back = __half22float2(hh);
                hi[nt][e] = *reinterpret_cast<const uint32_t*>(&hh);
                lo[nt][e] = pack_h2(v[2 * e] - back.x, v[2 * e + 1] - back.y);
            }
        }
#pragma unroll
        for (int mt = 0; mt < 4; mt++) {
            uint32_t a0[4], a1[4];
            load_a_fast<FMT>(st + aoff[t] + mt * 2048, a0, a1);
            const float s0 = scale_t<FMT>(sw0[mt], t), s1 = scale_t<FMT>(sw1[mt], t);
#pragma unroll
            for (int nt = 0; nt < NT; nt++) {
                {
                    float pp[4] = {0.f, 0.f, 0.f, 0.f};
                    mma_f16(pp, a0[0], a0[1], a0[2], a0[3], hi[nt][0], hi[nt][1]);
                    mma_f16(pp, a1[0], a1[1], a1[2], a1[3], hi[nt][2], hi[nt][3]);
                    mma_f16(pp, a0[0], a0[1], a0[2], a0[3], lo[nt][0], lo[nt][1]);
                    mma_f16(pp, a1[0], a1[1], a1[2], a1[3], lo[nt][2], lo[nt][3]);
                    fma4(acc[mt][nt], s0, s1, pp);
                }
            }
        }
    }
}

// the block rows behind pair column `col` of expert v
struct ItemCtx {
    int v, r, NT, pb, u_off;
    bool shared;
};

__device__ __forceinline__ int pair_row(const ExParams& p, const ItemCtx& c, int col) {
    return c.shared ? col : __ldg(p.pair + c.u_off + col) / p.top_k;
}

// f16 copy of one bf16 row scaled by 2^-p, p from the row's largest magnitude (the
// routing kernel's rule), by the EX_CT consumer threads: the row is held in
// registers between its max and its conversion (16-byte loads, all issued first).
constexpr int F16_ROW_PER = 4;  // 16-byte chunks per thread: rows of up to 8192 elements
__device__ void row_to_f16(int d, const uint16_t* __restrict__ x, __half* x16, int* xexp, uint32_t* s_max) {
    const int tid = threadIdx.x, nv = d / 8;
    const uint4* xv = reinterpret_cast<const uint4*>(x);
    uint4 v[F16_ROW_PER];
#pragma unroll
    for (int j = 0; j < F16_ROW_PER; j++) {
        const int c = j * EX_CT + tid;
        v[j] = c < nv ? __ldg(xv + c) : make_uint4(0, 0, 0, 0);
    }
    uint32_t mx = 0;
#pragma unroll
    for (int j = 0; j < F16_ROW_PER; j++) {
        const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
        for (int t = 0; t < 4; t++) mx = max(mx, max((w[t] & 0x7FFFu) << 16, w[t] & 0x7FFF0000u));
    }
    mx = __reduce_max_sync(0xffffffffu, mx);
    if ((tid & 31) == 0) s_max[tid >> 5] = mx;
    consumer_sync<EX_CT>();
    uint32_t m = 0;
#pragma unroll
    for (int w = 0; w < EX_CW; w++) m = max(m, s_max[w]);
    consumer_sync<EX_CT>();  // s_max is reused by the next row
    const int pe = f16_scale_exponent(m);
    const float sc = exp2i(-pe);
    uint4* ov = reinterpret_cast<uint4*>(x16);
#pragma unroll
    for (int j = 0; j < F16_ROW_PER; j++) {
        const int c = j * EX_CT + tid;
        if (c >= nv) continue;
        const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
        uint32_t o[4];
#pragma unroll
        for (int t = 0; t < 4; t++) {
            const __half2 h = __floats2half2_rn(__uint_as_float(w[t] << 16) * sc, __uint_as_float(w[t] & 0xFFFF0000u) * sc);
            o[t] = *reinterpret_cast<const uint32_t*>(&h);
        }
        ov[c] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (tid == 0) *xexp = pe;
}

// The shared-expert launch makes its own f16 copy of the block's rows: each CTA
// claims rows until none is left, then every CTA waits (bounded) until all rows
// are written.  Rows are claimed only by running CTAs, so the wait always ends.
__device__ void prepare_rows(const ExParams& p) {
    __shared__ uint32_t s_max[EX_CW];
    __shared__ int s_row;
    const int tid = threadIdx.x;
    __half* x16 = const_cast<__half*>(p.x16);
    int* xexp = const_cast<int*>(p.xexp);
    while (true) {
        if (tid == 0) s_row = (int)atomicAdd(p.ctrl + CTRL_PREP_SH, 1u);
        consumer_sync<EX_CT>();
        const int n = s_row;
        consumer_sync<EX_CT>();
        if (n >= p.n_rows) break;
        row_to_f16(p.k_gu, p.x_rows + (size_t)n * p.k_gu, x16 + (size_t)n * p.k_gu, xexp + n, s_max);
        __threadfence();
        consumer_sync<EX_CT>();
        if (tid == 0) red_release_add(p.ctrl + CTRL_PREPD_SH, 1u);
    }
    if (tid == 0 && ld_acquire(p.ctrl + CTRL_PREPD_SH) < (uint32_t)p.n_rows) {
        const uint64_t t0 = global_ns();
        while (ld_acquire(p.ctrl + CTRL_PREPD_SH) < (uint32_t)p.n_rows) {
            if (timed_out(p.ctrl)) break;
            if (global_ns() - t0 > WAIT_LIMIT_NS) {
                set_error(p.ctrl, MOE_EBIT_TIMEOUT);
                break;
            }
            __nanosleep(64);
        }
    }
    consumer_sync<EX_CT>();  // the copy is read with coherent (L1-cached, not .nc) loads
}

// ---------------------------------------------------------------------------

__device__ void producer(const ExParams& p, int V, unsigned char* ring, uint64_t* full, uint64_t* empty,
                         Meta* meta) {
    for (int m = 0; m < 12; m++) tma_prefetch_desc(&p.map[m]);
    const int S = p.n_shared;
    const int total = total_items(p, V);
    uint32_t stage = 0, phase = 0;
    uint32_t pending = 0, pending_par = 0;  // stages with copies not yet known to be consumed
    bool ok = true;
    while (ok) {
        const int item = (int)atomicAdd(p.ctrl + p.work_word, 1u);
        if (item >= total) break;
        int type, v, blk;
        decode_item(p, V, item, type, v, blk);
        const bool shared = v < S;
        const Geom& G = p.geom[(shared ? 2 : 0) + type];
        const CUtensorMap* mp = &p.map[shared ? 6 : 0];
        int z = v;
        if (!shared) {
            const int e = __ldg(p.uexp + ordered_index(p.uorder, v - S, V - S));
            z = __ldg(p.expert_slot + e);
            if (z < 0 || z >= p.n_slots) {
                set_error(p.ctrl, MOE_EBIT_BAD_SLOT);
                z = 0;
            }
            // gate/up items need the slot's gate/up planes (bit 0), down items its down planes (bit 1)
            const uint32_t need = type == IT_GU ? MOE_SLOT_GATE_UP : MOE_SLOT_DOWN;
            if (p.slot_ready != nullptr && (ld_acquire(p.slot_ready + z) & need) == 0u) {
                const uint64_t t0 = global_ns();
                while ((ld_acquire(p.slot_ready + z) & need) == 0u) {
                    // once any wait of this launch has run out, later ones give up at once
                    if (timed_out(p.ctrl)) break;
                    if (global_ns() - t0 > WAIT_LIMIT_NS) {
                        set_error(p.ctrl, MOE_EBIT_TIMEOUT);
                        break;
                    }
                    __nanosleep(256);
                }
            }
        }
        int rb = blk, c0 = 0, c1 = G.chunks;
        if (type == IT_DN && ksplit_of(p) > 1) {
            const int ks = ksplit_of(p);
            rb = blk / ks;
            const int r = blk - rb * ks;
            c0 = r * G.chunks / ks;
            c1 = (r + 1) * G.chunks / ks;
        }
        const int row0 = rb * G.rows_item;
        for (int c = c0; c < c1; c++) {
            if (!mbar_wait(&empty[stage], phase ^ 1u)) {
                set_error(p.ctrl, MOE_EBIT_TIMEOUT);
                ok = false;
                break;
            }
            pending &= ~(1u << stage);
            Meta& mt = meta[stage];
            mt.item = item;
            mt.type = type;
            mt.v = v;
            mt.blk = blk;
            mt.chunk = c;
            mt.nchunks = c1;
            mt.c0 = c0;
            mt.slot = z;
            mbar_arrive_expect_tx(&full[stage], G.tx);
            unsigned char* st = ring + (size_t)stage * EX_STAGE;
            if (G.merged) {
                // 16 KB of codes in one box ([matrix][K chunk][row][128 B], the layout
                // of the per-chunk boxes), the stage's scales in a second one
                if (type == IT_GU) {
                    tma_load_5d(st, mp, &full[stage], 0, row0, c * G.nbox, 0, z);
                    tma_load_4d(st + EX_CODE_BYTES, mp + 1, &full[stage], c * G.sb, row0, 0, z);
                } else {
                    tma_load_4d(st, mp + 4, &full[stage], 0, row0, c * G.nbox, z);
                    tma_load_3d(st + EX_CODE_BYTES, mp + 5, &full[stage], c * G.sb, row0, z);
                }
            } else if (type == IT_GU) {
                for (int m = 0; m < 2; m++) {
                    for (int b = 0; b < G.nbox; b++)
                        tma_load_3d(st + m * G.nbox * G.bi * 16 + b * G.bi * 16, mp + 2 * m, &full[stage],
                                    c * G.cb + b * G.bi, row0, z);
                    if (G.flat)
                        tma_load_3d(st + EX_CODE_BYTES + m * 512, mp + 2 * m + 1, &full[stage], 0,
                                    row0 * G.sb / 16, z);
                    else
                        tma_load_3d(st + EX_CODE_BYTES + m * 512, mp + 2 * m + 1, &full[stage], c * G.sb, row0, z);
                }
            } else {
                for (int b = 0; b < G.nbox; b++)
                    tma_load_3d(st + b * G.bi * 64, mp + 4, &full[stage], c * G.cb + b * G.bi, row0, z);
                if (G.flat)
                    tma_load_3d(st + EX_CODE_BYTES, mp + 5, &full[stage], 0, row0 * G.sb / 16, z);
                else
                    tma_load_3d(st + EX_CODE_BYTES, mp + 5, &full[stage], c * G.sb, row0, z);
            }
            pending |= 1u << stage;
            pending_par = (pending_par & ~(1u << stage)) | (phase << stage);
            if (++stage == EX_NST) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    if (ok) {
        if (mbar_wait(&empty[stage], phase ^ 1u)) {
            pending &= ~(1u << stage);
            meta[stage].item = -1;
            mbar_arrive(&full[stage]);
        } else {
            set_error(p.ctrl, MOE_EBIT_TIMEOUT);
        }
    }
    // never leave the CTA with copies in flight
    for (int s = 0; s < EX_NST; s++)
        if (pending & (1u << s)) mbar_wait(&full[s], (pending_par >> s) & 1u);
}

template <int FR, int FS, bool FAST>
__device__ void consumer(const ExParams& p, int V, const __half* x16, const int* xexp, bool x_global,
                         unsigned char* ring, float* red_base, uint64_t* full,
                         uint64_t* empty, const Meta* meta) {
    const int tid = threadIdx.x, cw = tid >> 5, lane = tid & 31;
    const int S = p.n_shared, N = p.n_rows;
    uint32_t stage = 0, phase = 0;
    ItemCtx c{};
    const __half* xrow[EX_NT];
    const float* hrow[EX_NT];
    float hs[EX_NT];
    bool bval[EX_NT];
    float acc[4][EX_NT][4];
    int type = IT_GU, blk = 0;
    uint32_t items_done = 0;
    // scale exponents of the h columns of the last expert whose down items ran here
    // (final once its gate/up items are done; the same for all its down items)
    __shared__ int s_hexp[EX_NT * 8];
    __shared__ int s_hexp_v;
    __shared__ int s_klast;  // this CTA finished the last K range of a split row block
    if (tid == 0) s_hexp_v = -1;
    consumer_sync<EX_CT>();

    while (true) {
        if (!mbar_wait(&full[stage], phase)) {
            if (lane == 0) set_error(p.ctrl, MOE_EBIT_TIMEOUT);
            break;
        }
        const Meta m = meta[stage];
        if (m.item < 0) break;
        if (m.chunk == m.c0) {
            type = m.type;
            blk = m.blk;
            c.v = m.v;
            c.shared = m.v < S;
            if (c.shared) {
                c.r = N;
                c.pb = m.v * N;
                c.u_off = 0;
            } else {
                const int u = ordered_index(p.uorder, m.v - S, V - S);
                const int o0 = __ldg(p.off + u), o1 = __ldg(p.off + u + 1);
                c.r = o1 - o0;
                c.pb = S * N + o0;
                c.u_off = o0;
            }
            c.NT = (c.r + 7) >> 3;
            if (c.NT > EX_NT) {
                if (lane == 0) set_error(p.ctrl, MOE_EBIT_BAD_SLOT);
                c.NT = EX_NT;
            }
#pragma unroll
            for (int nt = 0; nt < EX_NT; nt++) {
                const int col = nt * 8 + (lane >> 2);
                bval[nt] = col < c.r;
                xrow[nt] = x16;
                hrow[nt] = p.h;
                hs[nt] = 1.f;
                if (bval[nt]) {
                    if (type == IT_GU) {
                        xrow[nt] = x16 + (size_t)pair_row(p, c, col) * p.k_gu;
                    } else {
                        hrow[nt] = p.h + (size_t)(c.pb + col) * p.k_dn;
                    }
                }
#pragma unroll
                for (int t = 0; t < 4; t++) {
#pragma unroll
                    for (int mt = 0; mt < 4; mt++) acc[mt][nt][t] = 0.f;
                }
            }
            if (type == IT_DN) {
                if (p.job == J_LAYER) {
                    // the expert's gate/up items must be complete (bounded wait)
                    if (tid == 0 && ld_acquire(p.gu_done + c.v) < (uint32_t)p.n_gu) {
                        const uint64_t t0 = global_ns();
                        while (ld_acquire(p.gu_done + c.v) < (uint32_t)p.n_gu) {
                            if (timed_out(p.ctrl)) break;
                            if (global_ns() - t0 > WAIT_LIMIT_NS) {
                                set_error(p.ctrl, MOE_EBIT_TIMEOUT);
                                break;
                            }
                            __nanosleep(128);
                        }
                    }
                    consumer_sync<EX_CT>();
                }
                const int cached = s_hexp_v;
                consumer_sync<EX_CT>();
                if (cached != c.v) {
                    if (tid < c.r && tid < EX_NT * 8) s_hexp[tid] = f16_scale_exponent(__ldcg(p.hmax + c.pb + tid));
                    if (tid == 0) s_hexp_v = c.v;
                    consumer_sync<EX_CT>();
                }
#pragma unroll
                for (int nt = 0; nt < EX_NT; nt++)
                    if (bval[nt]) hs[nt] = exp2i(-s_hexp[nt * 8 + (lane >> 2)]);
                if constexpr (FAST) {  // the first stage's h lines (each stage prefetches the next)
                    const int T = c.shared ? Tiles<FS>::T_DN : Tiles<FR>::T_DN;
#pragma unroll
                    for (int nt = 0; nt < EX_NT; nt++)
                        if (bval[nt] && (lane & 3) < T)
                            asm volatile("prefetch.global.L1 [%0];" ::"l"(
                                hrow[nt] + (m.chunk * 8 * T + cw * T + (lane & 3)) * 32));
                }
            }
        }
        const uint32_t st = smem_u32(ring + (size_t)stage * EX_STAGE);
        if constexpr (FAST) {
            if (type == IT_GU) {
                if (c.shared) {
                    if (c.NT == 1)
                        gu_stage_fast<FS, Tiles<FS>::T_GU, 1>(st, m.chunk, m.nchunks, cw, lane, x_global, xrow, bval, acc[0], acc[1]);
                    else
                        gu_stage_fast<FS, Tiles<FS>::T_GU, 2>(st, m.chunk, m.nchunks, cw, lane, x_global, xrow, bval, acc[0], acc[1]);
                } else {
                    if (c.NT == 1)
                        gu_stage_fast<FR, Tiles<FR>::T_GU, 1>(st, m.chunk, m.nchunks, cw, lane, x_global, xrow, bval, acc[0], acc[1]);
                    else
                        gu_stage_fast<FR, Tiles<FR>::T_GU, 2>(st, m.chunk, m.nchunks, cw, lane, x_global, xrow, bval, acc[0], acc[1]);
                }
            } else {
                if (c.shared) {
                    if (c.NT == 1)
                        dn_stage_fast<FS, Tiles<FS>::T_DN, 1>(st, m.chunk, m.nchunks, cw, lane, hrow, hs, bval, acc);
                    else
                        dn_stage_fast<FS, Tiles<FS>::T_DN, 2>(st, m.chunk, m.nchunks, cw, lane, hrow, hs, bval, acc);
                } else {
                    if (c.NT == 1)
                        dn_stage_fast<FR, Tiles<FR>::T_DN, 1>(st, m.chunk, m.nchunks, cw, lane, hrow, hs, bval, acc);
                    else
                        dn_stage_fast<FR, Tiles<FR>::T_DN, 2>(st, m.chunk, m.nchunks, cw, lane, hrow, hs, bval, acc);
                }
            }
        } else {
            if (type == IT_GU) {
                if (c.shared)
                    gu_stage<FS>(st, p.geom[2], m.chunk, cw, lane, c.NT, xrow, bval, acc[0], acc[1]);
                else
                    gu_stage<FR>(st, p.geom[0], m.chunk, cw, lane, c.NT, xrow, bval, acc[0], acc[1]);
            } else {
                if (c.shared)
                    dn_stage<FS>(st, p.geom[3], m.chunk, cw, lane, c.NT, hrow, hs, bval, acc);
                else
                    dn_stage<FR>(st, p.geom[1], m.chunk, cw, lane, c.NT, hrow, hs, bval, acc);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);
        if (++stage == EX_NST) {
            stage = 0;
            phase ^= 1u;
        }
        if (m.chunk != m.nchunks - 1) continue;

        // ---- item epilogue: fixed-order reduction over the consumer warps ----
        // (two buffers alternate between items, so one barrier per item suffices
        // before the reads: a warp writing item i+1 cannot overwrite item i's data)
        float* red = red_base;
        if (type == IT_GU) {
            red = red_base + (items_done & 1u) * EX_RED_GU;
            items_done++;
#pragma unroll
            for (int nt = 0; nt < EX_NT; nt++)
#pragma unroll
                for (int t = 0; t < 4; t++) {
                    red[((cw * 2 + 0) * EX_NT + nt) * 128 + t * 32 + lane] = acc[0][nt][t];
                    red[((cw * 2 + 1) * EX_NT + nt) * 128 + t * 32 + lane] = acc[1][nt][t];
                }
            consumer_sync<EX_CT>();
            bool wrote = false;
            for (int idx = tid; idx < c.NT * 128; idx += EX_CT) {
                const int nt = idx >> 7, t = (idx >> 5) & 3, ln = idx & 31;
                float gs = 0.f, us = 0.f;
                for (int w = 0; w < EX_CW; w++) {
                    gs += red[((w * 2 + 0) * EX_NT + nt) * 128 + t * 32 + ln];
                    us += red[((w * 2 + 1) * EX_NT + nt) * 128 + t * 32 + ln];
                }
                const int col = nt * 8 + 2 * (ln & 3) + (t & 1);
                const int j = blk * 16 + (ln >> 2) + 8 * (t >> 1);
                uint32_t amax = 0;
                if (col < c.r) {
                    const int row = pair_row(p, c, col);
                    const float sc = exp2i(xexp[row]);
                    gs *= sc;
                    us *= sc;
                    const float hv = gs / (1.f + expf(-gs)) * us;
                    const size_t o = (size_t)(c.pb + col) * p.m_gu + j;
                    p.h[o] = hv;
                    if (p.debug_gu) {
                        p.dbg_g[o] = gs;
                        p.dbg_u[o] = us;
                    }
                    amax = __float_as_uint(hv) & 0x7FFFFFFFu;
                    wrote = true;
                }
                amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
                amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 8));
                amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 16));
                if (ln < 4 && col < c.r) atomicMax(p.hmax + c.pb + col, amax);
            }
            if (wrote) __threadfence();
            consumer_sync<EX_CT>();
            if (tid == 0) red_release_add(p.gu_done + c.v, 1u);
        } else {
            // the down item needs the whole buffer: wait for every reader of the last item
            consumer_sync<EX_CT>();
            items_done = 0;
#pragma unroll
            for (int mt = 0; mt < 4; mt++)
#pragma unroll
                for (int nt = 0; nt < EX_NT; nt++)
#pragma unroll
                    for (int t = 0; t < 4; t++) red[((cw * 4 + mt) * EX_NT + nt) * 128 + t * 32 + lane] = acc[mt][nt][t];
            consumer_sync<EX_CT>();
            const int ks = ksplit_of(p);
            const int rb = blk / ks, kr = blk - rb * ks;  // row block and K range of a split item
            const int per_mt = c.NT * 128;
            for (int idx = tid; idx < 4 * per_mt; idx += EX_CT) {
                const int mt = idx / per_mt, rem = idx - mt * per_mt;
                const int nt = rem >> 7, t = (rem >> 5) & 3, ln = rem & 31;
                const int col = nt * 8 + 2 * (ln & 3) + (t & 1);
                if (col >= c.r) continue;
                float y = 0.f;
                for (int w = 0; w < EX_CW; w++) y += red[((w * 4 + mt) * EX_NT + nt) * 128 + t * 32 + ln];
                y *= exp2i(s_hexp[col]);
                const int mrow = rb * 64 + mt * 16 + (ln >> 2) + 8 * (t >> 1);
                if (ks > 1) {
                    p.kpart[((size_t)kr * N + c.pb + col) * p.m_dn + mrow] = y;
                } else if (c.shared) {
                    float* dst = p.out_shared + (size_t)(c.pb + col) * p.m_dn + mrow;
                    *dst = p.accum ? (*dst + y) : y;
                } else {
                    const int pid = __ldg(p.pair + c.u_off + col);
                    p.y_part[(size_t)pid * p.m_dn + mrow] = y;
                }
            }
            if (ks > 1) {
                // the row block's last item to finish adds the K ranges' sums in range order
                __threadfence();
                consumer_sync<EX_CT>();
                if (tid == 0) s_klast = atomicAdd(p.karrive + rb, 1u) == (uint32_t)(ks - 1);
                consumer_sync<EX_CT>();
                if (s_klast) {
                    __threadfence();
                    for (int idx = tid; idx < c.r * 64; idx += EX_CT) {
                        const int col = idx >> 6, mrow = rb * 64 + (idx & 63);
                        const float* src = p.kpart + (size_t)(c.pb + col) * p.m_dn + mrow;
                        float y = __ldcg(src);
                        for (int r = 1; r < ks; r++) y += __ldcg(src + (size_t)r * N * p.m_dn);
                        float* dst = p.out_shared + (size_t)(c.pb + col) * p.m_dn + mrow;
                        *dst = p.accum ? (*dst + y) : y;
                    }
                }
            }
        }
    }
}

template <int FR, int FS, bool FAST>
__global__ void __launch_bounds__(EX_THREADS, 1) expert_kernel(const __grid_constant__ ExParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    unsigned char* ring = smem;
    float* red = reinterpret_cast<float*>(ring + (size_t)EX_NST * EX_STAGE);
    __half* xs = reinterpret_cast<__half*>(red + EX_RED_FLOATS);
    int* xs_exp = reinterpret_cast<int*>(reinterpret_cast<unsigned char*>(xs) + EX_XS_BYTES);  // [16]
    uint64_t* full = reinterpret_cast<uint64_t*>(xs_exp + 16);
    uint64_t* empty = full + EX_NST;
    Meta* meta = reinterpret_cast<Meta*>(empty + EX_NST);
    __shared__ int s_last;

    const int tid = threadIdx.x;
    const int tl_kernel = p.job == J_LAYER ? (p.routed_off ? TL_SHARED : TL_ROUTED) : -1;
    if (tid == 0 && tl_kernel >= 0) tl_begin(p.ctrl, tl_kernel);
    if (tid == 0) {
        for (int s = 0; s < EX_NST; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], EX_CW);
        }
        mbar_fence_init();
    }
    __syncthreads();
    // launched after the previous kernel on the stream: wait for it here, unless this
    // launch reads nothing that kernel writes (the shared experts beside the routing),
    // in which case it waits before it completes
    // the stand-alone Q8_0 jobs' producer reads only weights and this launch's work
    // counter, which the preparation kernel before it does not touch: it starts
    // streaming at once, and the consumers wait for the prepared rows
    const bool early_weights = p.job != J_LAYER && tid >= EX_CT;
    if (!p.dep_at_end && !early_weights) griddep_wait();
    griddep_launch_dependents();
    const int S = p.n_shared;
    const int U = (p.job == J_LAYER && !p.routed_off) ? (int)p.ctrl[CTRL_UNIQUE] : 0;
    const int V = S + U;

    if (tid >= EX_CT) {
        if (tid == EX_CT) producer(p, V, ring, full, empty, meta);
        return;
    }
    const __half* x16 = p.x16;
    const int* xexp = p.xexp;
    if (p.x_rows != nullptr && p.x_smem) {
        // every CTA makes the f16 copy it reads (no hand-off between CTAs)
        __shared__ uint32_t s_max[EX_CW];
        for (int n = 0; n < p.n_rows; n++)
            row_to_f16(p.k_gu, p.x_rows + (size_t)n * p.k_gu, xs + (size_t)n * p.k_gu, xs_exp + n, s_max);
        consumer_sync<EX_CT>();
        x16 = xs;
        xexp = xs_exp;
    } else if (p.x_rows != nullptr) {
        prepare_rows(p);
    }
    consumer<FR, FS, FAST>(p, V, x16, xexp, !(p.x_rows != nullptr && p.x_smem), ring, red, full, empty, meta);

    // the last CTA to finish leaves the workspace clean for the next call
    consumer_sync<EX_CT>();
    if (tid == 0) {
        __threadfence();
        s_last = atomicAdd(p.ctrl + p.exit_word, 1u) == gridDim.x - 1;
    }
    consumer_sync<EX_CT>();
    if (s_last) {
        __threadfence();
        for (int i = tid; i < V; i += EX_CT) p.gu_done[i] = 0;
        for (int64_t i = tid; i < p.pairs_cap; i += EX_CT) p.hmax[i] = 0;
        if (ksplit_of(p) > 1)
            for (int i = tid; i < p.n_dn; i += EX_CT) p.karrive[i] = 0;
        if (tid == 0) {
            p.ctrl[p.work_word] = 0;
            p.ctrl[p.exit_word] = 0;
            if (p.x_rows != nullptr && !p.x_smem) {
                p.ctrl[CTRL_PREP_SH] = 0;
                p.ctrl[CTRL_PREPD_SH] = 0;
            }
        }
    }
    if (tid == 0 && tl_kernel >= 0) tl_end(p.ctrl, tl_kernel);
    if (p.dep_at_end && tid == 0) griddep_wait();  // complete only after the previous kernel
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    // looked up once (thread-safe initialisation of a function-local static)
    static const EncodeTiledFn fn = [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(ptr);
        return static_cast<EncodeTiledFn>(nullptr);
    }();
    return fn;
}

static bool make_geom(Geom& g, int fmt, bool gu, int K, int rows_total) {
    g.rows_item = gu ? 16 : 64;
    g.row_bytes = fmt == MOE_FMT_MXFP4 ? K / 2 : K;
    const int cap = gu ? 512 : 256;
    g.cb = g.row_bytes < cap ? g.row_bytes : cap;
    if (g.cb <= 0 || g.row_bytes % g.cb) return false;
    g.bi = (g.cb % 128 == 0) ? 128 : g.cb;
    if (g.bi % 16 || g.bi > 128) return false;
    g.nbox = g.cb / g.bi;
    g.chunks = g.row_bytes / g.cb;
    g.gps = fmt == MOE_FMT_MXFP4 ? g.cb / 16 : g.cb / 32;
    g.sb = fmt == MOE_FMT_MXFP4 ? g.gps : 2 * g.gps;
    g.flat = g.sb < 16;
    const int rsb = (fmt == MOE_FMT_MXFP4 ? 1 : 2) * (K / 32);
    if (g.flat && (g.chunks != 1 || (g.rows_item * g.sb) % 16)) return false;
    if (!g.flat && rsb % 16) return false;
    if (rows_total % g.rows_item) return false;
    g.tx = (uint32_t)((gu ? 2 : 1) * (g.nbox * g.bi * g.rows_item + g.rows_item * g.sb));
    g.fast = (g.bi == 128 && g.cb == cap) ? 1 : 0;
    g.merged = 0;  // set by pool_maps with the maps it builds for fast stages
    return true;
}

// codes and scales maps of one [rows][K] matrix stored at `codes`/`scales`
// in each of n_slots slots slot_bytes apart
static bool make_maps(CUtensorMap* cm, CUtensorMap* sm, const Geom& g, int fmt, const void* codes,
                      const void* scales, int rows, int K, int n_slots, int64_t slot_bytes) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    if (((uintptr_t)codes & 15) || ((uintptr_t)scales & 15)) return false;
    const cuuint32_t estr[3] = {1, 1, 1};
    {
        const cuuint64_t dims[3] = {(cuuint64_t)g.row_bytes, (cuuint64_t)rows, (cuuint64_t)n_slots};
        const cuuint64_t strides[2] = {(cuuint64_t)g.row_bytes, (cuuint64_t)slot_bytes};
        const cuuint32_t box[3] = {(cuuint32_t)g.bi, (cuuint32_t)g.rows_item, 1};
        if (enc(cm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(codes), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, g.bi == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    const int rsb = (fmt == MOE_FMT_MXFP4 ? 1 : 2) * (K / 32);
    if (g.flat) {
        const cuuint64_t dims[3] = {16, (cuuint64_t)rows * rsb / 16, (cuuint64_t)n_slots};
        const cuuint64_t strides[2] = {16, (cuuint64_t)slot_bytes};
        const cuuint32_t box[3] = {16, (cuuint32_t)(g.rows_item * g.sb / 16), 1};
        return enc(sm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(scales), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }
    const cuuint64_t dims[3] = {(cuuint64_t)rsb, (cuuint64_t)rows, (cuuint64_t)n_slots};
    const cuuint64_t strides[2] = {(cuuint64_t)rsb, (cuuint64_t)slot_bytes};
    const cuuint32_t box[3] = {(cuuint32_t)g.sb, (cuuint32_t)g.rows_item, 1};
    return enc(sm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(scales), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// tiled uint8 map of rank 3 to 5: dims[0] contiguous, byte strides of dims 1..rank-1
static bool map_u8(CUtensorMap* m, const void* addr, int rank, const uint64_t* dims, const uint64_t* strides,
                   const uint32_t* box, bool swizzle) {
    EncodeTiledFn enc = encode_fn();
    if (!enc || rank < 3 || rank > 5 || ((uintptr_t)addr & 15)) return false;
    cuuint64_t gd[5], gs[4];
    cuuint32_t bx[5], es[5] = {1, 1, 1, 1, 1};
    for (int i = 0; i < rank; i++) {
        gd[i] = dims[i];
        bx[i] = box[i];
    }
    for (int i = 0; i + 1 < rank; i++) gs[i] = strides[i];
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, (cuuint32_t)rank, const_cast<void*>(addr), gd, gs, bx, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// all six maps of a slab pool (gate, up, down)
static bool pool_maps(CUtensorMap* maps, Geom* gg /*[2]: gate/up, down*/, const moe_pool* pool, int d, int f) {
    const int fmt = pool->format;
    if (!make_geom(gg[0], fmt, true, d, f) || !make_geom(gg[1], fmt, false, f, d)) return false;
    const char* base = static_cast<const char*>(pool->base);
    const int64_t cpb = fmt == MOE_FMT_MXFP4 ? 1 : 2;  // scale bytes per group
    const int64_t codes_gu = fmt == MOE_FMT_MXFP4 ? (int64_t)f * d / 2 : (int64_t)f * d;
    const int64_t scales_gu = (int64_t)f * (d / 32) * cpb;
    const int64_t per = codes_gu + scales_gu;
    if (gg[0].fast != gg[1].fast) gg[0].fast = gg[1].fast = 0;
    if (gg[0].fast) {
        // one box per stage and operand: gate and up codes [slot][matrix][row][K/128][128],
        // their scales [slot][matrix][row][K/32 groups], down codes [slot][row][K/128][128]
        const uint64_t sl = (uint64_t)pool->slot_bytes, ns = (uint64_t)pool->n_slots;
        const Geom& a = gg[0];
        const Geom& b = gg[1];
        const uint64_t rsb_gu = (uint64_t)cpb * (d / 32), rsb_dn = (uint64_t)cpb * (f / 32);
        {
            const uint64_t dims[5] = {128, (uint64_t)f, (uint64_t)a.row_bytes / 128, 2, ns};
            const uint64_t str[4] = {(uint64_t)a.row_bytes, 128, (uint64_t)per, sl};
            const uint32_t box[5] = {128, (uint32_t)a.rows_item, (uint32_t)a.nbox, 2, 1};
            if (!map_u8(&maps[0], base, 5, dims, str, box, true)) return false;
        }
        {
            const uint64_t dims[4] = {rsb_gu, (uint64_t)f, 2, ns};
            const uint64_t str[3] = {rsb_gu, (uint64_t)per, sl};
            const uint32_t box[4] = {(uint32_t)a.sb, (uint32_t)a.rows_item, 2, 1};
            if (!map_u8(&maps[1], base + codes_gu, 4, dims, str, box, false)) return false;
        }
        maps[2] = maps[0];
        maps[3] = maps[1];
        {
            const uint64_t dims[4] = {128, (uint64_t)d, (uint64_t)b.row_bytes / 128, ns};
            const uint64_t str[3] = {(uint64_t)b.row_bytes, 128, sl};
            const uint32_t box[4] = {128, (uint32_t)b.rows_item, (uint32_t)b.nbox, 1};
            if (!map_u8(&maps[4], base + 2 * per, 4, dims, str, box, true)) return false;
        }
        {
            const uint64_t dims[3] = {rsb_dn, (uint64_t)d, ns};
            const uint64_t str[2] = {rsb_dn, sl};
            const uint32_t box[3] = {(uint32_t)b.sb, (uint32_t)b.rows_item, 1};
            if (!map_u8(&maps[5], base + 2 * per + (fmt == MOE_FMT_MXFP4 ? (int64_t)d * f / 2 : (int64_t)d * f),
                        3, dims, str, box, false))
                return false;
        }
        gg[0].merged = gg[1].merged = 1;
        return true;
    }
    if (!make_maps(&maps[0], &maps[1], gg[0], fmt, base, base + codes_gu, f, d, pool->n_slots, pool->slot_bytes))
        return false;
    if (!make_maps(&maps[2], &maps[3], gg[0], fmt, base + per, base + per + codes_gu, f, d, pool->n_slots,
                   pool->slot_bytes))
        return false;
    return make_maps(&maps[4], &maps[5], gg[1], fmt, base + 2 * per, base + 2 * per + codes_gu, d, f, pool->n_slots,
                     pool->slot_bytes);
}

static int sm_count() {
    static const int n = [] {
        int dev = 0, v = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            v = 0;
        return v;
    }();
    return n;
}

template <int FR, int FS, bool FAST>
static int launch_variant(const ExParams& p, cudaStream_t stream) {
    static const cudaError_t attr = kernel_smem_attrs(expert_kernel<FR, FS, FAST>, (int)EX_SMEM);
    if (attr != cudaSuccess) return MOE_ERR_CUDA;
    const int grid = sm_count() * EX_CTAS_PER_SM;
    if (grid <= 0) return MOE_ERR_CUDA;
    if (launch_chained(expert_kernel<FR, FS, FAST>, dim3(grid), dim3(EX_THREADS), EX_SMEM, stream, p) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

// The unrolled fast paths serve every matrix of the job when all their stages
// are full width (the Kimi shapes); other shapes take the generic paths.
template <int FR, int FS>
static int launch_expert_kernel(const ExParams& p, cudaStream_t stream) {
    const bool fast = p.geom[0].fast && p.geom[1].fast && p.geom[2].fast && p.geom[3].fast;
    return fast ? launch_variant<FR, FS, true>(p, stream) : launch_variant<FR, FS, false>(p, stream);
}

}  // namespace moe

using namespace moe;

extern "C" int32_t moe_device_sm_count(void) { return sm_count(); }

extern "C" size_t moe_slab_bytes(const moe_desc* desc, int32_t format) {
    if (!desc) return 0;
    const size_t df = (size_t)desc->d_model * desc->d_ff;
    if (format == MOE_FMT_MXFP4) return 3 * (df / 2 + df / 32);
    if (format == MOE_FMT_Q8_0) return 3 * (df + 2 * (df / 32));
    return 0;
}

static bool pool_ok(const moe_desc* desc, const moe_pool* pool, int fmt) {
    if (!pool || !pool->base || pool->format != fmt || pool->n_slots <= 0) return false;
    if (((uintptr_t)pool->base & 31) || (pool->slot_bytes & 31)) return false;
    return (size_t)pool->slot_bytes >= moe_slab_bytes(desc, fmt);
}

extern "C" int moe_expert_block(const moe_desc* desc, int32_t n_rows, int32_t mode, const moe_pool* routed,
                                const int32_t* expert_slot, const uint32_t* slot_ready, const moe_pool* shared,
                                int32_t n_shared, void* ws, int32_t n_rows_max, float* y_part, void* stream) {
    if (!desc || !ws || !expert_slot || !y_part) return MOE_ERR_INVALID_ARG;
    const int d = desc->d_model, f = desc->d_ff, E = desc->n_experts, k = desc->top_k;
    if (desc->group != 32 || d <= 0 || d % 256 || f <= 0 || f % 64 || E <= 0 || E > 1024 || k < 1 || k > 32 || k > E)
        return MOE_ERR_UNSUPPORTED;
    const int base_mode = mode & 0xFF;
    if (base_mode != MOE_MODE_DECODE && base_mode != MOE_MODE_PREFILL) return MOE_ERR_UNSUPPORTED;
    const bool only_shared = (mode & MOE_MODE_SHARED_ONLY) != 0, only_routed = (mode & MOE_MODE_ROUTED_ONLY) != 0;
    if (only_shared && only_routed) return MOE_ERR_INVALID_ARG;
    if ((mode & MOE_MODE_AFTER_SHARED) && !only_routed) return MOE_ERR_INVALID_ARG;
    if (n_rows < 1 || n_rows > n_rows_max) return MOE_ERR_UNSUPPORTED;
    if (base_mode == MOE_MODE_DECODE && n_rows > 16) return MOE_ERR_UNSUPPORTED;
    // blocks of more than 16 rows: routed experts on the block-scaled path only (the
    // shared experts' engine serves up to 16 rows)
    if (n_rows > 16 && (!tc_expert_supported(d, f, n_rows) || only_shared || (n_shared > 0 && !only_routed)))
        return MOE_ERR_UNSUPPORTED;
    if (n_shared < 0 || n_shared > 8) return MOE_ERR_UNSUPPORTED;
    if (!pool_ok(desc, routed, MOE_FMT_MXFP4)) return MOE_ERR_INVALID_ARG;
    if (n_shared > 0 && (!pool_ok(desc, shared, MOE_FMT_Q8_0) || shared->n_slots < n_shared)) return MOE_ERR_INVALID_ARG;
    if ((uintptr_t)ws & 255) return MOE_ERR_INVALID_ARG;

    const WsLayout L = ws_layout(d, f, E, k, n_rows_max, n_shared);
    char* base = static_cast<char*>(ws);
    thread_local ExParams p;  // large (tensor maps); filled per call, copied into the launch
    memset(&p, 0, sizeof(p));
    if (!pool_maps(&p.map[0], &p.geom[0], routed, d, f)) return MOE_ERR_UNSUPPORTED;
    if (n_shared > 0 && !pool_maps(&p.map[6], &p.geom[2], shared, d, f)) return MOE_ERR_UNSUPPORTED;
    if (n_shared == 0) {
        for (int i = 0; i < 6; i++) p.map[6 + i] = p.map[i];
        p.geom[2] = p.geom[0];
        p.geom[3] = p.geom[1];
    }
    p.job = J_LAYER;
    p.fmt_routed = MOE_FMT_MXFP4;
    p.fmt_shared = MOE_FMT_Q8_0;
    p.k_gu = d;
    p.m_gu = f;
    p.k_dn = f;
    p.m_dn = d;
    p.top_k = k;
    p.n_rows = n_rows;
    p.n_shared = n_shared;
    p.n_gu = f / 16;
    p.n_dn = d / 64;
    p.lag = 4;
    p.debug_gu = (mode & MOE_MODE_DEBUG_GU) ? 1 : 0;
    p.accum = 0;
    p.expert_slot = expert_slot;
    p.slot_ready = slot_ready;
    p.n_slots = routed->n_slots;
    p.ctrl = reinterpret_cast<uint32_t*>(base + L.ctrl);
    p.uexp = reinterpret_cast<const int*>(base + L.uexp);
    p.off = reinterpret_cast<const int*>(base + L.off);
    p.uorder = (mode & MOE_MODE_ORDERED) ? reinterpret_cast<const int*>(base + L.uorder) : nullptr;
    p.pair = reinterpret_cast<const int*>(base + L.pair);
    p.x16 = reinterpret_cast<const __half*>(base + L.x16);
    p.xexp = reinterpret_cast<const int*>(base + L.xexp);
    p.gu_done = reinterpret_cast<uint32_t*>(base + L.gu_done);
    p.hmax = reinterpret_cast<uint32_t*>(base + L.hmax);
    p.h = reinterpret_cast<float*>(base + L.h);
    p.dbg_g = reinterpret_cast<float*>(base + L.dbg_g);
    p.dbg_u = reinterpret_cast<float*>(base + L.dbg_u);
    p.out_shared = reinterpret_cast<float*>(base + L.shared_y);
    p.y_part = y_part;
    p.pairs_cap = L.pairs;
    p.work_word = CTRL_WORK;
    p.exit_word = CTRL_EXIT;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (only_shared && n_shared == 0) return MOE_OK;
    if (tc_expert_supported(d, f, n_rows)) {
        // shared Q8_0 experts on the tensor-core MMA.sync engine, routed MXFP4
        // experts on the block-scaled tcgen05 kernel
        if (n_shared > 0 && !only_routed) {
            p.routed_off = 1;
            const int st = launch_expert_kernel<MOE_FMT_MXFP4, MOE_FMT_Q8_0>(p, s);
            if (st != MOE_OK || only_shared) return st;
        }
        return tc_expert_launch(desc, n_rows, mode, routed, expert_slot, slot_ready, n_shared, ws, n_rows_max, y_part,
                                s);
    }
    if (only_shared) p.routed_off = 1;
    if (only_routed) p.n_shared = 0;
    return launch_expert_kernel<MOE_FMT_MXFP4, MOE_FMT_Q8_0>(p, s);
}

static int shared_experts(const moe_desc* desc, int32_t n_rows, const uint16_t* x, const moe_pool* shared,
                          int32_t n_shared, void* ws, int32_t n_rows_max, bool after_route, void* stream) {
    if (!desc || !ws || !x || !shared) return MOE_ERR_INVALID_ARG;
    const int d = desc->d_model, f = desc->d_ff, E = desc->n_experts, k = desc->top_k;
    if (desc->group != 32 || d <= 0 || d % 256 || f <= 0 || f % 64 || E <= 0 || E > 1024 || k < 1 || k > 32 || k > E)
        return MOE_ERR_UNSUPPORTED;
    if (n_rows < 1 || n_rows > n_rows_max) return MOE_ERR_UNSUPPORTED;
    if (n_shared < 1 || n_shared > 8) return MOE_ERR_UNSUPPORTED;
    if (!pool_ok(desc, shared, MOE_FMT_Q8_0) || shared->n_slots < n_shared) return MOE_ERR_INVALID_ARG;
    if (((uintptr_t)ws & 255) || ((uintptr_t)x & 15)) return MOE_ERR_INVALID_ARG;
    // blocks of more than 16 rows (prefill): the register-streaming kernels of shared.cu
    if (n_rows > 16)
        return shared_launch(desc, n_rows, n_rows_max, x, shared, n_shared, ws, true, !after_route,
                             static_cast<cudaStream_t>(stream));
    if (d > F16_ROW_PER * EX_CT * 8) return MOE_ERR_UNSUPPORTED;

    const WsLayout L = ws_layout(d, f, E, k, n_rows_max, n_shared);
    char* base = static_cast<char*>(ws);
    thread_local ExParams p;  // filled per call, copied into the launch
    memset(&p, 0, sizeof(p));
    if (!pool_maps(&p.map[6], &p.geom[2], shared, d, f)) return MOE_ERR_UNSUPPORTED;
    for (int i = 0; i < 6; i++) p.map[i] = p.map[6 + i];  // no routed experts in this launch
    p.geom[0] = p.geom[2];
    p.geom[1] = p.geom[3];
    p.job = J_LAYER;
    p.fmt_routed = MOE_FMT_MXFP4;
    p.fmt_shared = MOE_FMT_Q8_0;
    p.k_gu = d;
    p.m_gu = f;
    p.k_dn = f;
    p.m_dn = d;
    p.top_k = k;
    p.n_rows = n_rows;
    p.n_shared = n_shared;
    p.n_gu = f / 16;
    p.n_dn = d / 64;
    p.lag = 4;
    p.routed_off = 1;
    p.n_slots = 1;
    p.ctrl = reinterpret_cast<uint32_t*>(base + L.ctrl);
    p.x16 = reinterpret_cast<const __half*>(base + L.x16s);
    p.xexp = reinterpret_cast<const int*>(base + L.xexps);
    p.gu_done = reinterpret_cast<uint32_t*>(base + L.gu_done_sh);
    p.hmax = reinterpret_cast<uint32_t*>(base + L.hmax_sh);
    p.h = reinterpret_cast<float*>(base + L.h_sh);  // shared pairs: rows [0, n_shared * N)
    p.out_shared = reinterpret_cast<float*>(base + L.shared_y);
    p.pairs_cap = (int64_t)n_shared * n_rows_max;
    p.work_word = CTRL_WORK_SH;
    p.exit_word = CTRL_EXIT_SH;
    p.x_rows = x;
    // rows in device memory: every CTA makes its own f16 copy in shared memory (from
    // L2).  Rows in host memory (read in place over the host link): one CTA makes the
    // copy in the workspace and the others wait for it, so the rows cross the link
    // once rather than once per CTA.  The copy is the same either way.
    cudaPointerAttributes pa{};
    const cudaError_t qe = cudaPointerGetAttributes(&pa, x);
    if (qe != cudaSuccess) (void)cudaGetLastError();  // a failed query leaves no error behind
    const bool x_host = qe == cudaSuccess && pa.type == cudaMemoryTypeHost;
    p.x_smem = !x_host && (size_t)n_rows * d * 2 <= (size_t)EX_XS_BYTES ? 1 : 0;
    p.dep_at_end = after_route ? 1 : 0;
    return launch_expert_kernel<MOE_FMT_MXFP4, MOE_FMT_Q8_0>(p, static_cast<cudaStream_t>(stream));
}

extern "C" int moe_shared_experts(const moe_desc* desc, int32_t n_rows, const uint16_t* x, const moe_pool* shared,
                                  int32_t n_shared, void* ws, int32_t n_rows_max, void* stream) {
    return shared_experts(desc, n_rows, x, shared, n_shared, ws, n_rows_max, false, stream);
}

extern "C" int moe_shared_experts_after_route(const moe_desc* desc, int32_t n_rows, const uint16_t* x,
                                              const moe_pool* shared, int32_t n_shared, void* ws, int32_t n_rows_max,
                                              void* stream) {
    return shared_experts(desc, n_rows, x, shared, n_shared, ws, n_rows_max, true, stream);
}

// ---------------------------------------------------------------------------
// stand-alone Q8_0 block matmul
// ---------------------------------------------------------------------------

struct Q8Ws {
    size_t ctrl, x16, xexp, hmax, h, gu_done, kpart, karrive, karrive_bytes, total;
};

// K ranges of the plain job's 64-row down items.  Unsplit, a narrow projection has
// only n_out / 64 items for the whole GPU (7168 -> 1536: 24 items on 152 SMs, each
// streaming 7168 bytes of codes for 64 rows), so most SMs stay idle; split into ks
// ranges it has n_dn * ks items of about C / ks chunks (C = k_in / 256 chunks of 64
// rows x 256 bytes).  ks minimises ceil(items / SMs) * (chunks per item + 1), the + 1
// standing for an item's partial store and hand-over.  It depends on the shape and
// the SM count, never on n_rows, so a row's result is the same in every block.  At
// most Q8_KSPLIT_ELEMS / n_out ranges, which bounds the partial sums' scratch.
constexpr int Q8_KSPLIT_MAX = 32;
constexpr int Q8_KSPLIT_ELEMS = 32768;  // ks * n_out

static int q8_ksplit_cap(int k_in, int n_out) {
    int cap = Q8_KSPLIT_ELEMS / n_out;
    cap = std::min(cap, k_in / 256);
    cap = std::min(cap, Q8_KSPLIT_MAX);
    return cap >= 2 ? cap : 1;
}

static int q8_ksplit(int k_in, int n_out, int n_sm) {
    const int C = k_in / 256, n_dn = n_out / 64, cap = q8_ksplit_cap(k_in, n_out);
    int best = 1;
    int64_t best_cost = (int64_t)((n_dn + n_sm - 1) / n_sm) * C;
    for (int ks = 2; ks <= cap; ks++) {
        const int64_t cost = (int64_t)((n_dn * ks + n_sm - 1) / n_sm) * ((C + ks - 1) / ks + 1);
        if (cost < best_cost) {
            best = ks;
            best_cost = cost;
        }
    }
    return best;
}

static Q8Ws q8_layout(int n_rows, int k_in, int n_out) {
    Q8Ws L;
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 256); return at; };
    L.ctrl = take(CTRL_WORDS * 4);
    L.x16 = take((size_t)n_rows * k_in * 2);
    L.xexp = take((size_t)n_rows * 4);
    L.hmax = take((size_t)n_rows * 4);
    L.h = take((size_t)n_rows * k_in * 4);
    L.gu_done = take(4);
    // partial sums and arrival counters of split down items (plain job), sized for the
    // largest split the shape allows
    const int cap = q8_ksplit_cap(k_in, n_out);
    L.kpart = cap > 1 ? take((size_t)cap * n_rows * n_out * 4) : 0;
    L.karrive_bytes = cap > 1 ? (size_t)(n_out / 64) * 4 : 0;
    L.karrive = cap > 1 ? take(L.karrive_bytes) : 0;
    L.total = o;
    return L;
}

// prepares the rows of a stand-alone Q8_0 matmul: f16 rows (SwiGLU) or fp32 rows
// with their largest magnitude (plain).  One CTA per row; each thread loads all its
// 8-element pieces of a pass before it uses any of them, so a row costs one or two
// memory round trips instead of one per element.  It lets the matmul kernel launch
// at once: that kernel's producer streams weights (which this kernel does not touch)
// while its consumers wait for these rows.
constexpr int Q8P_THREADS = 512;
constexpr int Q8P_UNROLL = 2;  // 8-element pieces per thread and pass

__device__ __forceinline__ void q8p_load8(const void* __restrict__ x, int x_dtype, bool vec, size_t i,
                                          float (&v)[8]) {
    if (x_dtype == MOE_DTYPE_BF16) {
        const uint16_t* xb = static_cast<const uint16_t*>(x) + i;
        if (vec) {
            const uint4 u = __ldg(reinterpret_cast<const uint4*>(xb));
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; e++) {
                v[2 * e] = __uint_as_float(w[e] << 16);
                v[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
            }
        } else {
#pragma unroll
            for (int e = 0; e < 8; e++) v[e] = __uint_as_float((uint32_t)__ldg(xb + e) << 16);
        }
    } else {
        const float* xf = static_cast<const float*>(x) + i;
        if (vec) {
            const float4 a = __ldg(reinterpret_cast<const float4*>(xf));
            const float4 b = __ldg(reinterpret_cast<const float4*>(xf + 4));
            v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w, v[4] = b.x, v[5] = b.y, v[6] = b.z, v[7] = b.w;
        } else {
#pragma unroll
            for (int e = 0; e < 8; e++) v[e] = __ldg(xf + e);
        }
    }
}

__global__ void __launch_bounds__(Q8P_THREADS) q8_prep_kernel(int k_in, const void* __restrict__ x, int x_dtype,
                                                              int swiglu, int vec, __half* __restrict__ x16,
                                                              int* __restrict__ xexp, uint32_t* __restrict__ hmax,
                                                              float* __restrict__ h) {
    griddep_launch_dependents();
    const int n = blockIdx.x, tid = threadIdx.x;
    __shared__ uint32_t s_max[Q8P_THREADS / 32];
    __shared__ int s_p;
    const size_t row = (size_t)n * k_in;
    constexpr int PASS = Q8P_THREADS * 8 * Q8P_UNROLL;
    uint32_t mx = 0;
    for (int c0 = 0; c0 < k_in; c0 += PASS) {
        float v[Q8P_UNROLL][8];
#pragma unroll
        for (int u = 0; u < Q8P_UNROLL; u++) {
            const int c = c0 + (u * Q8P_THREADS + tid) * 8;  // k_in % 256 == 0: all 8 in range
            if (c < k_in) q8p_load8(x, x_dtype, vec != 0, row + c, v[u]);
        }
#pragma unroll
        for (int u = 0; u < Q8P_UNROLL; u++) {
            const int c = c0 + (u * Q8P_THREADS + tid) * 8;
            if (c >= k_in) continue;
#pragma unroll
            for (int e = 0; e < 8; e++) mx = max(mx, __float_as_uint(v[u][e]) & 0x7FFFFFFFu);
            if (!swiglu) {
                float4* dst = reinterpret_cast<float4*>(h + row + c);
                dst[0] = make_float4(v[u][0], v[u][1], v[u][2], v[u][3]);
                dst[1] = make_float4(v[u][4], v[u][5], v[u][6], v[u][7]);
            }
        }
    }
    for (int o = 16; o; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((tid & 31) == 0) s_max[tid >> 5] = mx;
    __syncthreads();
    if (tid == 0) {
        uint32_t m = 0;
        for (int w = 0; w < Q8P_THREADS / 32; w++) m = max(m, s_max[w]);
        s_p = f16_scale_exponent(m);
        hmax[n] = m;
        xexp[n] = s_p;
    }
    __syncthreads();
    if (swiglu) {
        const float sc = exp2i(-s_p);
        for (int c0 = 0; c0 < k_in; c0 += PASS) {
            float v[Q8P_UNROLL][8];
#pragma unroll
            for (int u = 0; u < Q8P_UNROLL; u++) {
                const int c = c0 + (u * Q8P_THREADS + tid) * 8;
                if (c < k_in) q8p_load8(x, x_dtype, vec != 0, row + c, v[u]);
            }
#pragma unroll
            for (int u = 0; u < Q8P_UNROLL; u++) {
                const int c = c0 + (u * Q8P_THREADS + tid) * 8;
                if (c >= k_in) continue;
                __half2 hv[4];
#pragma unroll
                for (int e = 0; e < 4; e++)
                    hv[e] = __halves2half2(__float2half_rn(v[u][2 * e] * sc), __float2half_rn(v[u][2 * e + 1] * sc));
                *reinterpret_cast<uint4*>(x16 + row + c) = *reinterpret_cast<const uint4*>(hv);
            }
        }
    }
}

extern "C" size_t q8_0_workspace_size(int32_t n_rows, int32_t k_in, int32_t n_out) {
    if (n_rows <= 0 || k_in <= 0 || n_out <= 0) return 0;
    return q8_layout(n_rows, k_in, n_out).total;
}

extern "C" int q8_0_block_matmul(int32_t n_rows, int32_t k_in, int32_t n_out, const void* x, int32_t x_dtype,
                                 const int8_t* q, const uint16_t* dq, const int8_t* q2, const uint16_t* d2,
                                 int32_t epilogue, float* y, void* ws, void* stream) {
    if (!x || !q || !dq || !y || !ws) return MOE_ERR_INVALID_ARG;
    if (n_rows < 1 || n_rows > 16 || k_in <= 0 || k_in % 256 || n_out <= 0) return MOE_ERR_UNSUPPORTED;
    if (x_dtype != MOE_DTYPE_BF16 && x_dtype != MOE_DTYPE_F32) return MOE_ERR_INVALID_ARG;
    const bool swiglu = epilogue == MOE_EPI_SWIGLU;
    if (!swiglu && epilogue != MOE_EPI_NONE && epilogue != MOE_EPI_ACCUM) return MOE_ERR_INVALID_ARG;
    if (swiglu && (!q2 || !d2 || x_dtype != MOE_DTYPE_BF16)) return MOE_ERR_INVALID_ARG;
    if (swiglu ? (n_out % 16) : (n_out % 64)) return MOE_ERR_UNSUPPORTED;
    if (((uintptr_t)q & 31) || ((uintptr_t)dq & 31) || ((uintptr_t)ws & 255)) return MOE_ERR_INVALID_ARG;
    if (swiglu && (((uintptr_t)q2 & 31) || ((uintptr_t)d2 & 31))) return MOE_ERR_INVALID_ARG;

    const Q8Ws L = q8_layout(n_rows, k_in, n_out);
    char* base = static_cast<char*>(ws);
    thread_local ExParams p;  // filled per call, copied into the launch
    memset(&p, 0, sizeof(p));
    Geom g;
    if (!make_geom(g, MOE_FMT_Q8_0, swiglu, k_in, n_out)) return MOE_ERR_UNSUPPORTED;
    const int64_t qbytes = align_up((size_t)n_out * k_in, 32);
    const int64_t dbytes = align_up((size_t)n_out * (k_in / 32) * 2, 32);
    const int64_t slot = qbytes > dbytes ? qbytes : dbytes;
    if (swiglu) {
        if (!make_maps(&p.map[6], &p.map[7], g, MOE_FMT_Q8_0, q, dq, n_out, k_in, 1, slot)) return MOE_ERR_UNSUPPORTED;
        if (!make_maps(&p.map[8], &p.map[9], g, MOE_FMT_Q8_0, q2, d2, n_out, k_in, 1, slot)) return MOE_ERR_UNSUPPORTED;
        p.map[10] = p.map[6];
        p.map[11] = p.map[7];
        p.geom[2] = g;
        p.geom[3] = g;
        p.job = J_Q8_SWIGLU;
    } else {
        if (!make_maps(&p.map[10], &p.map[11], g, MOE_FMT_Q8_0, q, dq, n_out, k_in, 1, slot)) return MOE_ERR_UNSUPPORTED;
        p.map[6] = p.map[8] = p.map[10];
        p.map[7] = p.map[9] = p.map[11];
        p.geom[2] = g;
        p.geom[3] = g;
        p.job = J_Q8_PLAIN;
    }
    for (int i = 0; i < 6; i++) p.map[i] = p.map[6 + i];
    p.geom[0] = p.geom[2];
    p.geom[1] = p.geom[3];
    p.fmt_routed = p.fmt_shared = MOE_FMT_Q8_0;
    p.k_gu = k_in;
    p.m_gu = n_out;
    p.k_dn = k_in;
    p.m_dn = n_out;
    p.top_k = 1;
    p.n_rows = n_rows;
    p.n_shared = 1;
    p.n_gu = n_out / 16;
    p.n_dn = n_out / 64;
    p.lag = 0;
    p.accum = epilogue == MOE_EPI_ACCUM;
    p.n_slots = 1;
    p.ctrl = reinterpret_cast<uint32_t*>(base + L.ctrl);
    p.x16 = reinterpret_cast<const __half*>(base + L.x16);
    p.xexp = reinterpret_cast<const int*>(base + L.xexp);
    p.gu_done = reinterpret_cast<uint32_t*>(base + L.gu_done);
    p.hmax = reinterpret_cast<uint32_t*>(base + L.hmax);
    p.h = swiglu ? y : reinterpret_cast<float*>(base + L.h);
    p.out_shared = y;
    p.dbg_g = p.dbg_u = nullptr;
    p.pairs_cap = 0;  // hmax rows are rewritten by the preparation kernel on every call
    p.work_word = CTRL_WORK;
    p.exit_word = CTRL_EXIT;
    if (!swiglu) {
        p.ksplit = q8_ksplit(k_in, n_out, sm_count());
        if (p.ksplit > q8_ksplit_cap(k_in, n_out)) return MOE_ERR_UNSUPPORTED;
        p.kpart = reinterpret_cast<float*>(base + L.kpart);
        p.karrive = reinterpret_cast<uint32_t*>(base + L.karrive);
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int vec = ((uintptr_t)x & 15) == 0;  // rows are then 16-byte aligned too (k_in % 256 == 0)
    q8_prep_kernel<<<n_rows, Q8P_THREADS, 0, s>>>(k_in, x, x_dtype, swiglu ? 1 : 0, vec,
                                                  reinterpret_cast<__half*>(base + L.x16),
                                                  reinterpret_cast<int*>(base + L.xexp),
                                                  reinterpret_cast<uint32_t*>(base + L.hmax),
                                                  reinterpret_cast<float*>(base + L.h));
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
    return launch_expert_kernel<MOE_FMT_Q8_0, MOE_FMT_Q8_0>(p, s);
}

// ---------------------------------------------------------------------------
// stand-alone Q8_0 block matmul without any device allocation by the caller
// ---------------------------------------------------------------------------
//
// Some callers cannot allocate device memory for the scratch that
// q8_0_block_matmul needs: a host process that hands every byte of HBM to its
// own pool allocator up front, or a latency-critical serving path where a
// cudaMalloc/cudaFree (which can synchronise the device) is not acceptable.
// This variant takes its scratch from a file-scope __device__ array instead.
// The array lives in every GPU that loads this library until the process exits.

constexpr int Q8_NOALLOC_MAX_ROWS = 16;
constexpr int Q8_NOALLOC_MAX_K = 7168;
// >= q8_layout(16, 7168, n_out).total for every n_out: 689,408 bytes of rows and
// control words, at most 16 x Q8_KSPLIT_ELEMS floats of partial sums and 1 KB of
// arrival counters (a split needs n_out <= Q8_KSPLIT_ELEMS / 2), rounded to 4 KB
constexpr size_t Q8_NOALLOC_BYTES = 2789376;
constexpr int Q8_NOALLOC_MAX_DEVICES = 64;

static __device__ __align__(256) unsigned char q8_noalloc_scratch[Q8_NOALLOC_BYTES];

// Device address of the scratch array on each device, looked up with that device
// current (in host code the symbol's name is only a stand-in, not a device
// address).  The address belongs to the context it was looked up in: a device
// reset or a new primary context makes it stale, so the context is kept beside it
// and a change of context repeats the lookup.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

static CtxGetCurrentFn ctx_get_current_fn() {
    static const CtxGetCurrentFn fn = [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            return reinterpret_cast<CtxGetCurrentFn>(ptr);
        return static_cast<CtxGetCurrentFn>(nullptr);
    }();
    return fn;
}

struct NoallocSlot {
    std::mutex m;
    CUcontext ctx = nullptr;
    void* addr = nullptr;
};
static NoallocSlot q8_noalloc_slot[Q8_NOALLOC_MAX_DEVICES];

// The scratch array's device address on the current device (nullptr on failure).
static unsigned char* q8_noalloc_scratch_addr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= Q8_NOALLOC_MAX_DEVICES) return nullptr;
    CtxGetCurrentFn get_ctx = ctx_get_current_fn();
    CUcontext ctx = nullptr;
    if (!get_ctx || get_ctx(&ctx) != CUDA_SUCCESS) return nullptr;
    if (ctx == nullptr) {
        // no context current on this thread yet: the symbol lookup makes the
        // device's primary context current
        void* addr = nullptr;
        if (cudaGetSymbolAddress(&addr, q8_noalloc_scratch) != cudaSuccess) return nullptr;
        if (get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) return nullptr;
    }
    NoallocSlot& slot = q8_noalloc_slot[dev];
    std::lock_guard<std::mutex> lock(slot.m);
    if (slot.ctx != ctx || slot.addr == nullptr) {
        void* addr = nullptr;
        if (cudaGetSymbolAddress(&addr, q8_noalloc_scratch) != cudaSuccess || addr == nullptr) return nullptr;
        slot.ctx = ctx;
        slot.addr = addr;
    }
    return static_cast<unsigned char*>(slot.addr);
}

extern "C" int q8_0_block_matmul_noalloc(int32_t n_rows, int32_t k_in, int32_t n_out, const void* x,
                                         int32_t x_dtype, const int8_t* q, const uint16_t* dq, const int8_t* q2,
                                         const uint16_t* d2, int32_t epilogue, float* y, void* stream) {
    if (n_rows < 1 || n_rows > Q8_NOALLOC_MAX_ROWS || k_in <= 0 || k_in > Q8_NOALLOC_MAX_K)
        return MOE_ERR_UNSUPPORTED;
    const Q8Ws L = q8_layout(n_rows, k_in, n_out);
    if (L.total > Q8_NOALLOC_BYTES) return MOE_ERR_UNSUPPORTED;
    unsigned char* ws = q8_noalloc_scratch_addr();
    if (ws == nullptr) return MOE_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the array keeps the previous call's contents: clear the control words after the
    // error word (which collects the device errors of every call until
    // q8_0_noalloc_get_error reads and clears it) and the gate/up completion counter,
    // which the kernel expects to start at zero
    if (cudaMemsetAsync(ws + L.ctrl + 4 * (CTRL_ERROR + 1), 0, (CTRL_WORDS - CTRL_ERROR - 1) * 4, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (cudaMemsetAsync(ws + L.gu_done, 0, 4, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (L.karrive_bytes && cudaMemsetAsync(ws + L.karrive, 0, L.karrive_bytes, s) != cudaSuccess) return MOE_ERR_CUDA;
    return q8_0_block_matmul(n_rows, k_in, n_out, x, x_dtype, q, dq, q2, d2, epilogue, y, ws, stream);
}

extern "C" int q8_0_noalloc_get_error(void* stream, uint32_t* bits) {
    if (!bits) return MOE_ERR_INVALID_ARG;
    unsigned char* ws = q8_noalloc_scratch_addr();
    if (ws == nullptr) return MOE_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t* word = reinterpret_cast<uint32_t*>(ws) + CTRL_ERROR;  // the control block starts the array
    if (cudaMemcpyAsync(bits, word, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemsetAsync(word, 0, 4, s) != cudaSuccess) return MOE_ERR_CUDA;
    return cudaStreamSynchronize(s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
