// Shared experts (Q8_0) of prefill blocks (more than 16 rows): every row runs the
// same SwiGLU MLP with weights q * fp16(d) (int8, one fp16 scale per 32 along K).
//
// Pages: "Run Kimi K3 and K3.1 Pro Locally" (computingforgeeks.com), table in
// "Kimi K3 and K3.1 Pro in numbers" (16 of 896 routed experts plus 2 shared);
// "Run Kimi 3.1 locally on one GPU", sections "One GPU, three storage tiers"
// (the non-expert weights in Q8_0) and "A drafter that leaves the answer
// unchanged" (the spine's matrix multiplies load each weight once for all rows).
//
// Design (GB300): the weights stream straight from global memory into the
// registers of tensor-core fragments (no shared-memory staging, no producer
// warp); a gate/up warp works on 32 block rows at a time and a down warp on 16, so
// the weights are read from HBM once and from L2 for every further chunk of rows.  Decode blocks
// (up to 16 rows) use the TMA-fed engine of experts.cu instead, whose deeper
// staging keeps more bytes in flight per SM.
//
//   sh_prep_kernel  f16 copy of the block's rows, each scaled by a power of two
//                   2^-p chosen from the row's largest magnitude
//   sh_gu_kernel    gate and up projections: a warp owns 16 rows of gate and the
//                   same 16 rows of up, for 32 block rows, over one of SH_KS K
//                   slices; per 32-wide K group two m16n8k16 MMAs (f16 in, fp32
//                   out) give the group's exact partial, scaled by its fp16 scale
//                   into the accumulator; the last slice of a tile to finish sums
//                   the slices in slice order and applies SwiGLU (fp32 h)
//   sh_split_kernel h split once into f16 hi + lo parts (per-row power-of-two scale)
//   sh_dn_kernel    down projection: a warp owns 16 output rows and 16 block rows
//                   over the full K, on the hi and lo parts of h
//
// A thread (g = lane / 4, i = lane % 4) loads 8 consecutive int8 codes of its
// rows g and g + 8 per group (bytes 8i..8i+7): inside the group, K positions
// 8i+{0,1,2,3} and 8i+{4,5,6,7} play the fragment roles of K = {2i, 2i+1,
// 2i+8, 2i+9} of the group's first and second MMA.  The activations use the same
// assignment (thread (g, i) supplies bytes 8i..8i+7 of row g), so every product
// q[o][c] x[n][c] is formed exactly once.  A row's arithmetic never depends on
// the other rows of the block (MMA columns are independent; the K order is fixed).
#include "common.cuh"

namespace moe {
namespace sh {

constexpr int WARPS = 4;             // warps per CTA
constexpr int THREADS = WARPS * 32;
constexpr int SH_KS = SH_K_SPLIT;    // K slices of the gate/up projection
constexpr int UNROLL = 4;            // K groups whose loads are in flight together (down)
constexpr int GU_NT = 4;             // n-tiles (8 block rows each) of a gate/up warp unit
constexpr int GU_W = 8 * GU_NT;      // block rows of a gate/up warp unit
constexpr int GU_UNROLL = 3;         // K groups whose loads are in flight together (gate/up)

struct Params {
    const int8_t* q;          // shared pool base (slot s at q + s * slot_bytes)
    int64_t slot_bytes;
    int d, f, n_rows, n_shared, n_chunks;  // n_chunks = ceil(n_rows / 16): the down projection's row chunks
    int n_gchunks;                          // ceil(n_rows / GU_W): the gate/up projection's
    const __half* x16;        // [N][d] f16 rows (x * 2^-xexp)
    const int* xexp;          // [N]
    float* part;              // gate/up partials [s][tile][chunk][ks][2][16 rows][GU_W cols]
    uint32_t* cnt;            // [s][tile][chunk] slices finished
    float* h;                 // [s][N][f]
    __half* h_hi;             // [s][N][f] f16 parts of h * 2^-p (p from the row's max |h|): hi
    __half* h_lo;             // and lo = h * 2^-p - hi, rounded to f16
    uint32_t* hmax;           // [s][N] max |h| bits
    float* out;               // [s][N][d]
    uint32_t* ctrl;
    const uint16_t* x;        // bf16 rows for sh_prep_kernel
    __half* x16w;
    int* xexpw;
    int wait_at_start;        // programmatic dependent launch: wait before reading x16
    int wait_at_end;          // sh_prep_kernel: complete only after the previous kernel
};

__device__ __forceinline__ uint2 ldg64(const void* p) { return __ldg(reinterpret_cast<const uint2*>(p)); }

// fragment registers of one group: the 8 codes of row g (w0) and of row g + 8 (w1)
// -> A of the group's first MMA (a1) and second MMA (a2)
__device__ __forceinline__ void frags(uint2 w0, uint2 w1, uint32_t (&a1)[4], uint32_t (&a2)[4]) {
    uint32_t r0lo, r0hi, r0lo2, r0hi2, r1lo, r1hi, r1lo2, r1hi2;
    s8x4_to_f16x2(w0.x, r0lo, r0hi);   // row g: K 8i..8i+1, 8i+2..8i+3
    s8x4_to_f16x2(w0.y, r0lo2, r0hi2); // row g: K 8i+4..8i+5, 8i+6..8i+7
    s8x4_to_f16x2(w1.x, r1lo, r1hi);
    s8x4_to_f16x2(w1.y, r1lo2, r1hi2);
    a1[0] = r0lo; a1[1] = r1lo; a1[2] = r0hi; a1[3] = r1hi;
    a2[0] = r0lo2; a2[1] = r1lo2; a2[2] = r0hi2; a2[3] = r1hi2;
}

__device__ __forceinline__ float f16s(const uint16_t* p) { return __half2float(__ushort_as_half(__ldg(p))); }

// f16 copy of the block's rows: one CTA per row, x * 2^-p with p from the row's
// largest magnitude (max * 2^-p in [2^14, 2^15))
__global__ void __launch_bounds__(256) sh_prep_kernel(const Params p) {
    if (threadIdx.x == 0) tl_begin(p.ctrl, TL_SHARED);
    if (p.wait_at_start) griddep_wait();
    griddep_launch_dependents();
    const int n = blockIdx.x, tid = threadIdx.x;
    __shared__ uint32_t s_max[8];
    __shared__ int s_p;
    const uint16_t* x = p.x + (size_t)n * p.d;
    uint32_t mx = 0;
    for (int c = tid * 8; c < p.d; c += 256 * 8) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + c));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int t = 0; t < 4; t++) mx = max(mx, max((w[t] & 0x7FFFu) << 16, w[t] & 0x7FFF0000u));
    }
    mx = __reduce_max_sync(0xffffffffu, mx);
    if ((tid & 31) == 0) s_max[tid >> 5] = mx;
    __syncthreads();
    if (tid == 0) {
        uint32_t m = 0;
        for (int w = 0; w < 8; w++) m = max(m, s_max[w]);
        s_p = f16_scale_exponent(m);
        p.xexpw[n] = s_p;
        for (int s = 0; s < p.n_shared; s++) p.hmax[(size_t)s * p.n_rows + n] = 0u;
    }
    __syncthreads();
    const float sc = exp2i(-s_p);
    for (int c = tid * 8; c < p.d; c += 256 * 8) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + c));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int t = 0; t < 4; t++) {
            const __half2 h = __floats2half2_rn(__uint_as_float(w[t] << 16) * sc, __uint_as_float(w[t] & 0xFFFF0000u) * sc);
            o[t] = *reinterpret_cast<const uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>(p.x16w + (size_t)n * p.d + c) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (p.wait_at_end && tid == 0) griddep_wait();
}

// The loads of a window of GU_UNROLL K groups (weights, their scales, the activation
// fragments) are issued one window ahead of its MMAs: a warp keeps two windows in
// registers, so every global load has a window's worth of MMAs to hide behind.
struct GuWin {
    uint2 wg0[GU_UNROLL], wg1[GU_UNROLL], wu0[GU_UNROLL], wu1[GU_UNROLL];
    uint16_t sg0[GU_UNROLL], sg1[GU_UNROLL], su0[GU_UNROLL], su1[GU_UNROLL];
    uint4 x[GU_NT][GU_UNROLL];
};

// gate/up: warp unit = (expert s, 16-row tile, chunk of GU_W block rows, K slice).  The
// weights a warp converts to f16 serve all GU_NT n-tiles of its chunk.
__global__ void __launch_bounds__(THREADS) sh_gu_kernel(const Params p) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, i = lane & 3;
    const int tiles = p.f / 16;
    const int64_t units = (int64_t)p.n_shared * tiles * p.n_gchunks * SH_KS;
    const int64_t u = (int64_t)blockIdx.x * WARPS + warp;
    if (threadIdx.x == 0 && blockIdx.x == 0) tl_begin(p.ctrl, TL_SHARED);
    if (u >= units) {
        griddep_launch_dependents();
        return;
    }
    const int ks = (int)(u % SH_KS);
    const int64_t r1 = u / SH_KS;
    const int ch = (int)(r1 % p.n_gchunks);
    const int64_t r2 = r1 / p.n_gchunks;
    const int tile = (int)(r2 % tiles), s = (int)(r2 / tiles);
    const int d = p.d, f = p.f, ksl = d / SH_KS, G = ksl / 32;
    const int8_t* slab = p.q + (size_t)s * p.slot_bytes;
    const size_t per = (size_t)f * d + (size_t)f * (d / 32) * 2;  // one gate or up matrix with its scales
    const int o0 = tile * 16 + g;
    const int8_t* qg0 = slab + (size_t)o0 * d;
    const int8_t* qg1 = qg0 + (size_t)8 * d;
    const int8_t* qu0 = qg0 + per;
    const int8_t* qu1 = qg1 + per;
    const uint16_t* sg0 = reinterpret_cast<const uint16_t*>(slab + (size_t)f * d) + (size_t)o0 * (d / 32);
    const uint16_t* sg1 = sg0 + (size_t)8 * (d / 32);
    const uint16_t* su0 = reinterpret_cast<const uint16_t*>(reinterpret_cast<const int8_t*>(sg0) + per);
    const uint16_t* su1 = su0 + (size_t)8 * (d / 32);
    const int kbase = ks * ksl;
    const int nb = ch * GU_W;
    const int ntu = min(GU_NT, (p.n_rows - nb + 7) / 8);  // n-tiles of the chunk in use
    const __half* xr[GU_NT];  // B column (block row) nb + 8 nt + g of each n-tile
    bool xv[GU_NT];
#pragma unroll
    for (int nt = 0; nt < GU_NT; nt++) {
        const int n = nb + nt * 8 + g;
        xv[nt] = n < p.n_rows;
        xr[nt] = p.x16 + (size_t)(xv[nt] ? n : 0) * d;
    }
    auto load_w = [&](GuWin& w, int j0) {  // weights and scales of window j0 (independent of the rows)
#pragma unroll
        for (int t = 0; t < GU_UNROLL; t++) {
            const int j = j0 + t;
            if (j < G) {
                const int k = kbase + 32 * j;
                w.wg0[t] = ldg64(qg0 + k + 8 * i); w.wg1[t] = ldg64(qg1 + k + 8 * i);
                w.wu0[t] = ldg64(qu0 + k + 8 * i); w.wu1[t] = ldg64(qu1 + k + 8 * i);
                w.sg0[t] = __ldg(sg0 + k / 32); w.sg1[t] = __ldg(sg1 + k / 32);
                w.su0[t] = __ldg(su0 + k / 32); w.su1[t] = __ldg(su1 + k / 32);
            }
        }
    };
    auto load_x = [&](GuWin& w, int j0) {
#pragma unroll
        for (int t = 0; t < GU_UNROLL; t++) {
            const int k = kbase + 32 * (j0 + t) + 8 * i;
            const bool in = j0 + t < G;
#pragma unroll
            for (int nt = 0; nt < GU_NT; nt++)
                w.x[nt][t] = (in && nt < ntu && xv[nt]) ? __ldg(reinterpret_cast<const uint4*>(xr[nt] + k))
                                                        : make_uint4(0, 0, 0, 0);
        }
    };
    GuWin cur, nxt;
    load_w(cur, 0);  // requested before waiting for the rows
    if (p.wait_at_start) griddep_wait();
    griddep_launch_dependents();
    load_x(cur, 0);
    float ag[GU_NT][4], au[GU_NT][4];
#pragma unroll
    for (int nt = 0; nt < GU_NT; nt++)
#pragma unroll
        for (int t = 0; t < 4; t++) ag[nt][t] = au[nt][t] = 0.f;
    for (int j0 = 0; j0 < G; j0 += GU_UNROLL) {
        if (j0 + GU_UNROLL < G) {
            load_w(nxt, j0 + GU_UNROLL);
            load_x(nxt, j0 + GU_UNROLL);
        }
#pragma unroll
        for (int t = 0; t < GU_UNROLL; t++) {
            if (j0 + t >= G) break;
            uint32_t ga1[4], ga2[4], ua1[4], ua2[4];
            frags(cur.wg0[t], cur.wg1[t], ga1, ga2);
            frags(cur.wu0[t], cur.wu1[t], ua1, ua2);
            const float fg0 = __half2float(__ushort_as_half(cur.sg0[t])), fg1 = __half2float(__ushort_as_half(cur.sg1[t]));
            const float fu0 = __half2float(__ushort_as_half(cur.su0[t])), fu1 = __half2float(__ushort_as_half(cur.su1[t]));
#pragma unroll
            for (int nt = 0; nt < GU_NT; nt++) {
                if (nt >= ntu) break;
                const uint4 bx = cur.x[nt][t];
                float pg[4] = {0.f, 0.f, 0.f, 0.f}, pu[4] = {0.f, 0.f, 0.f, 0.f};
                mma_f16(pg, ga1[0], ga1[1], ga1[2], ga1[3], bx.x, bx.y);
                mma_f16(pg, ga2[0], ga2[1], ga2[2], ga2[3], bx.z, bx.w);
                mma_f16(pu, ua1[0], ua1[1], ua1[2], ua1[3], bx.x, bx.y);
                mma_f16(pu, ua2[0], ua2[1], ua2[2], ua2[3], bx.z, bx.w);
                ag[nt][0] = fmaf(fg0, pg[0], ag[nt][0]); ag[nt][1] = fmaf(fg0, pg[1], ag[nt][1]);
                ag[nt][2] = fmaf(fg1, pg[2], ag[nt][2]); ag[nt][3] = fmaf(fg1, pg[3], ag[nt][3]);
                au[nt][0] = fmaf(fu0, pu[0], au[nt][0]); au[nt][1] = fmaf(fu0, pu[1], au[nt][1]);
                au[nt][2] = fmaf(fu1, pu[2], au[nt][2]); au[nt][3] = fmaf(fu1, pu[3], au[nt][3]);
            }
        }
        cur = nxt;
    }
    // this slice's sums: part[tile unit][ks][gate|up][16 rows][GU_W cols]
    constexpr int UN = 16 * GU_W;  // sums of one matrix in one unit
    const int64_t tu = ((int64_t)s * tiles + tile) * p.n_gchunks + ch;
    float* dst = p.part + (tu * SH_KS + ks) * 2 * UN;
#pragma unroll
    for (int nt = 0; nt < GU_NT; nt++) {
        const int c = nt * 8 + 2 * i;
        dst[g * GU_W + c] = ag[nt][0];
        dst[g * GU_W + c + 1] = ag[nt][1];
        dst[(g + 8) * GU_W + c] = ag[nt][2];
        dst[(g + 8) * GU_W + c + 1] = ag[nt][3];
        dst[UN + g * GU_W + c] = au[nt][0];
        dst[UN + g * GU_W + c + 1] = au[nt][1];
        dst[UN + (g + 8) * GU_W + c] = au[nt][2];
        dst[UN + (g + 8) * GU_W + c + 1] = au[nt][3];
    }
    __threadfence();
    __syncwarp();
    uint32_t last = 0;
    if (lane == 0) last = atomicAdd(p.cnt + tu, 1u) == (uint32_t)(SH_KS - 1);
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) return;
    __threadfence();
    // the tile's last slice: sum the slices in slice order, then SwiGLU
    const float* src = p.part + tu * SH_KS * 2 * UN;
    for (int e = lane; e < UN; e += 32) {
        const int row = e / GU_W, col = e - row * GU_W, n = nb + col;
        if (n >= p.n_rows) continue;
        float gs = 0.f, us = 0.f;
#pragma unroll
        for (int q = 0; q < SH_KS; q++) {
            gs += __ldcg(src + q * 2 * UN + e);
            us += __ldcg(src + q * 2 * UN + UN + e);
        }
        const float sc = exp2i(__ldg(p.xexp + n));
        gs *= sc;
        us *= sc;
        const float hv = gs / (1.f + expf(-gs)) * us;
        p.h[((size_t)s * p.n_rows + n) * f + tile * 16 + row] = hv;
        atomicMax(p.hmax + (size_t)s * p.n_rows + n, __float_as_uint(hv) & 0x7FFFFFFFu);
    }
    if (lane == 0) p.cnt[tu] = 0u;
}

// h of every (shared expert, row) -> f16 hi + lo parts of h * 2^-p, p from the row's
// largest |h|: one CTA per (expert, row).  Each value is split once here instead of
// once per 16-row output tile of the down projection.
__global__ void __launch_bounds__(256) sh_split_kernel(const Params p) {
    griddep_wait();  // h and its row maxima come from the gate/up kernel
    griddep_launch_dependents();
    const size_t row = blockIdx.x;  // s * n_rows + n
    const float sc = exp2i(-f16_scale_exponent(__ldcg(p.hmax + row)));
    const float* h = p.h + row * p.f;
    for (int c = threadIdx.x * 4; c < p.f; c += 256 * 4) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(h + c));
        const float vv[4] = {v.x * sc, v.y * sc, v.z * sc, v.w * sc};
        uint32_t hi[2], lo[2];
#pragma unroll
        for (int e = 0; e < 2; e++) {
            const __half2 h2 = __floats2half2_rn(vv[2 * e], vv[2 * e + 1]);
            const float2 back = __half22float2(h2);
            hi[e] = *reinterpret_cast<const uint32_t*>(&h2);
            const __half2 l2 = __floats2half2_rn(vv[2 * e] - back.x, vv[2 * e + 1] - back.y);
            lo[e] = *reinterpret_cast<const uint32_t*>(&l2);
        }
        *reinterpret_cast<uint2*>(p.h_hi + row * p.f + c) = make_uint2(hi[0], hi[1]);
        *reinterpret_cast<uint2*>(p.h_lo + row * p.f + c) = make_uint2(lo[0], lo[1]);
    }
}

struct DnWin {
    uint2 w0[UNROLL], w1[UNROLL];
    uint16_t s0[UNROLL], s1[UNROLL];
    uint4 hi[2][UNROLL], lo[2][UNROLL];  // 8 f16 of each part per n-tile and group
};

// down: warp unit = (expert s, 16 output rows, 16-row chunk of the block), full K
__global__ void __launch_bounds__(THREADS) sh_dn_kernel(const Params p) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, i = lane & 3;
    const int tiles = p.d / 16;
    const int64_t units = (int64_t)p.n_shared * tiles * p.n_chunks;
    const int64_t u = (int64_t)blockIdx.x * WARPS + warp;
    if (u >= units) {
        griddep_wait();
        griddep_launch_dependents();
        return;
    }
    const int ch = (int)(u % p.n_chunks);
    const int64_t r1 = u / p.n_chunks;
    const int tile = (int)(r1 % tiles), s = (int)(r1 / tiles);
    const int d = p.d, f = p.f, G = f / 32;
    const int8_t* slab = p.q + (size_t)s * p.slot_bytes;
    const size_t per = (size_t)f * d + (size_t)f * (d / 32) * 2;
    const int o0 = tile * 16 + g;
    const int8_t* q0 = slab + 2 * per + (size_t)o0 * f;
    const int8_t* q1 = q0 + (size_t)8 * f;
    const uint16_t* s0 = reinterpret_cast<const uint16_t*>(slab + 2 * per + (size_t)d * f) + (size_t)o0 * (f / 32);
    const uint16_t* s1 = s0 + (size_t)8 * (f / 32);
    const int nb = ch * 16;
    // B columns this thread supplies (g, 8 + g) and C columns it holds (2i, 2i+1, 8+2i, 9+2i)
    const int nl = nb + g, nh = nb + 8 + g;
    const bool vl = nl < p.n_rows, vh = nh < p.n_rows;
    const bool two = nb + 8 < p.n_rows;
    const size_t rl = ((size_t)s * p.n_rows + (vl ? nl : 0)) * f, rh = ((size_t)s * p.n_rows + (vh ? nh : 0)) * f;
    auto load_w = [&](DnWin& w, int j0) {
#pragma unroll
        for (int t = 0; t < UNROLL; t++) {
            const int j = j0 + t;
            if (j < G) {
                w.w0[t] = ldg64(q0 + 32 * j + 8 * i);
                w.w1[t] = ldg64(q1 + 32 * j + 8 * i);
                w.s0[t] = __ldg(s0 + j);
                w.s1[t] = __ldg(s1 + j);
            }
        }
    };
    auto load_h = [&](DnWin& w, int j0) {
#pragma unroll
        for (int t = 0; t < UNROLL; t++) {
            const int k = 32 * (j0 + t) + 8 * i;
            const bool in = j0 + t < G;
#pragma unroll
            for (int nt = 0; nt < 2; nt++) {
                const bool v = in && (nt ? (two && vh) : vl);
                const size_t r = (nt ? rh : rl) + k;
                w.hi[nt][t] = v ? __ldg(reinterpret_cast<const uint4*>(p.h_hi + r)) : make_uint4(0, 0, 0, 0);
                w.lo[nt][t] = v ? __ldg(reinterpret_cast<const uint4*>(p.h_lo + r)) : make_uint4(0, 0, 0, 0);
            }
        }
    };
    DnWin cur, nxt;
    load_w(cur, 0);
    griddep_wait();  // the split parts of h come from the split kernel
    griddep_launch_dependents();
    load_h(cur, 0);
    float acc[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; nt++)
#pragma unroll
        for (int t = 0; t < 4; t++) acc[nt][t] = 0.f;
    for (int j0 = 0; j0 < G; j0 += UNROLL) {
        if (j0 + UNROLL < G) {
            load_w(nxt, j0 + UNROLL);
            load_h(nxt, j0 + UNROLL);
        }
#pragma unroll
        for (int t = 0; t < UNROLL; t++) {
            if (j0 + t >= G) break;
            uint32_t a1[4], a2[4];
            frags(cur.w0[t], cur.w1[t], a1, a2);
            const float fs0 = __half2float(__ushort_as_half(cur.s0[t])), fs1 = __half2float(__ushort_as_half(cur.s1[t]));
#pragma unroll
            for (int nt = 0; nt < 2; nt++) {
                if (nt == 1 && !two) break;
                const uint4 hv = cur.hi[nt][t], lv = cur.lo[nt][t];
                const uint32_t hi[4] = {hv.x, hv.y, hv.z, hv.w}, lo[4] = {lv.x, lv.y, lv.z, lv.w};
                float pp[4] = {0.f, 0.f, 0.f, 0.f};
                mma_f16(pp, a1[0], a1[1], a1[2], a1[3], hi[0], hi[1]);
                mma_f16(pp, a2[0], a2[1], a2[2], a2[3], hi[2], hi[3]);
                mma_f16(pp, a1[0], a1[1], a1[2], a1[3], lo[0], lo[1]);
                mma_f16(pp, a2[0], a2[1], a2[2], a2[3], lo[2], lo[3]);
                acc[nt][0] = fmaf(fs0, pp[0], acc[nt][0]);
                acc[nt][1] = fmaf(fs0, pp[1], acc[nt][1]);
                acc[nt][2] = fmaf(fs1, pp[2], acc[nt][2]);
                acc[nt][3] = fmaf(fs1, pp[3], acc[nt][3]);
            }
        }
        cur = nxt;
    }
#pragma unroll
    for (int nt = 0; nt < 2; nt++) {
#pragma unroll
        for (int e = 0; e < 2; e++) {
            const int n = nb + nt * 8 + 2 * i + e;
            if (n >= p.n_rows) continue;
            const float up = exp2i(f16_scale_exponent(__ldcg(p.hmax + (size_t)s * p.n_rows + n)));
            float* o = p.out + ((size_t)s * p.n_rows + n) * d + tile * 16;
            o[g] = acc[nt][e] * up;
            o[g + 8] = acc[nt][2 + e] * up;
        }
    }
    if (threadIdx.x == 0) tl_end(p.ctrl, TL_SHARED);
}

}  // namespace sh

// The shared experts of a block of n_rows rows from the f16 rows x16/xexp (written by
// the routing kernel for blocks of up to 32 rows, or by sh_prep_kernel from x):
// gate/up then down, chained with programmatic dependent launch.  prep: run the
// preparation kernel from x first.  wait_first: the first launch waits for the
// previous kernel on the stream before it reads anything.
int shared_launch(const moe_desc* desc, int n_rows, int n_rows_max, const uint16_t* x, const moe_pool* shared,
                  int n_shared, void* ws, bool prep, bool wait_first, cudaStream_t s) {
    using namespace sh;
    const int d = desc->d_model, f = desc->d_ff;
    if (d % (32 * SH_KS) || f % 32 || d % 16 || f % 16) return MOE_ERR_UNSUPPORTED;
    const WsLayout L = ws_layout(d, f, desc->n_experts, desc->top_k, n_rows_max, n_shared);
    char* base = static_cast<char*>(ws);
    Params p;
    memset(&p, 0, sizeof(p));
    p.q = static_cast<const int8_t*>(shared->base);
    p.slot_bytes = shared->slot_bytes;
    p.d = d;
    p.f = f;
    p.n_rows = n_rows;
    p.n_shared = n_shared;
    p.n_chunks = (n_rows + 15) / 16;
    p.n_gchunks = (n_rows + GU_W - 1) / GU_W;
    p.x16 = reinterpret_cast<const __half*>(base + (prep ? L.x16s : L.x16));
    p.xexp = reinterpret_cast<const int*>(base + (prep ? L.xexps : L.xexp));
    p.part = reinterpret_cast<float*>(base + L.sh_part);
    p.cnt = reinterpret_cast<uint32_t*>(base + L.sh_cnt);
    p.h = reinterpret_cast<float*>(base + L.h_sh);
    p.h_hi = reinterpret_cast<__half*>(base + L.h_sh_hl);
    p.h_lo = p.h_hi + (size_t)(n_shared > 0 ? n_shared : 1) * n_rows_max * f;
    p.hmax = reinterpret_cast<uint32_t*>(base + L.hmax_sh);
    p.out = reinterpret_cast<float*>(base + L.shared_y);
    p.ctrl = reinterpret_cast<uint32_t*>(base + L.ctrl);
    p.x = x;
    p.x16w = reinterpret_cast<__half*>(base + L.x16s);
    p.xexpw = reinterpret_cast<int*>(base + L.xexps);
    if (prep) {
        // wait_first: stream order for x; otherwise (right after moe_route, which reads
        // the same x) the preparation overlaps the routing and completes after it
        p.wait_at_start = wait_first ? 1 : 0;
        p.wait_at_end = wait_first ? 0 : 1;
        if (launch_chained(sh_prep_kernel, dim3(n_rows), dim3(256), 0, s, p) != cudaSuccess) return MOE_ERR_CUDA;
        p.wait_at_start = 1;
        p.wait_at_end = 0;
    } else {
        // the rows' maxima are gathered fresh for this block
        if (cudaMemsetAsync(p.hmax, 0, (size_t)n_shared * n_rows * 4, s) != cudaSuccess) return MOE_ERR_CUDA;
        p.wait_at_start = 1;
    }
    const int64_t gu_units = (int64_t)n_shared * (f / 16) * p.n_gchunks * SH_KS;
    const int64_t dn_units = (int64_t)n_shared * (d / 16) * p.n_chunks;
    if (launch_chained(sh_gu_kernel, dim3((unsigned)((gu_units + WARPS - 1) / WARPS)), dim3(THREADS), 0, s, p) !=
        cudaSuccess)
        return MOE_ERR_CUDA;
    if (launch_chained(sh_split_kernel, dim3((unsigned)(n_shared * n_rows)), dim3(256), 0, s, p) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (launch_chained(sh_dn_kernel, dim3((unsigned)((dn_units + WARPS - 1) / WARPS)), dim3(THREADS), 0, s, p) !=
        cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

}  // namespace moe
