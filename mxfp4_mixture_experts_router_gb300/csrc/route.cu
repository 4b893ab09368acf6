// Routing of a block of rows: router GEMV, top-k selection, renormalised
// weights, grouping of the block's (row, slot) pairs by expert, and the
// activation preparation the expert kernel reads.
//
// Pages: "Run Kimi 3.1 locally on one GPU", section "Read the experts the
// router needs" (16 of 896 experts per token); the router matrix is BF16
// ("Run Kimi K3 and K3.1 Pro Locally", section "Confirm the checkpoint format
// and size").  Softmax-then-renormalise over the selected k, ties to the
// lower index, is this library's reading of the unstated router function.
//
// One launch.  CTAs (kslice, egroup) each compute partial logits over a 512-wide
// K slice for 64 experts and all rows (every weight byte is loaded once, all
// loads issued up front); the last CTA of an expert group sums the K slices in
// slice order; the last group finisher selects the top-k of every row, forms
// the weights and groups the pairs.  Every logit is a fixed-order fp32 sum, so
// a row's logits, selection and weights do not depend on the other rows.
#include "common.cuh"

namespace moe {

constexpr int RT_THREADS = 256;
constexpr int RT_KS = 512;      // K elements per slice
constexpr int RT_EG = 64;       // experts per group (8 per warp)
constexpr int RT_MAX_ROWS = 32;
constexpr int RT_MAX_KS = 16;   // K slices: d <= 8192
constexpr int RT_TICKET_EG = 32;  // ctrl words [32, 64) hold the per-group tickets

struct RouteParams {
    int d, E, k, N, n_shared;
    int n_ks, n_eg, n_gemv_ctas;
    const uint16_t* x;
    const uint16_t* w;
    const float* logits_in;
    float* logits;        // logits_out, or the workspace copy
    float* part;          // [n_ks][N][E] partial logits
    int32_t* topk_idx;
    float* topk_w;
    uint32_t* ctrl;
    int* uexp;
    int* off;
    int* pair;
    __half* x16;
    int* xexp;
    uint32_t* gu_done;
    uint32_t* hmax;
    uint8_t* x_mx;        // [3N][d] E4M3 terms of x for the block-scaled expert kernel
    uint8_t* x_sc;        // [3N][d/32] their E8M0 scales
    uint32_t* gu_done_tc;
    int v_cap;
    int64_t pairs_cap;
};

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Activation preparation for the expert kernel: x16 = f16(x * 2^-p), p chosen
// from the row's largest magnitude so the row sits inside the f16 range.  Rows of
// up to 8192 elements stay in registers between the max and the conversion (all
// 16-byte loads issued before any is used); longer rows are read twice.
__device__ void prep_row(const uint16_t* x, int d, __half* x16, int* xexp, float* red) {
    constexpr int PER = 4;  // 16-byte chunks per thread and pass
    const int tid = threadIdx.x;
    const int nv = d / 8;
    const uint4* xv = reinterpret_cast<const uint4*>(x);
    uint4* ov = reinterpret_cast<uint4*>(x16);
    const bool resident = nv <= PER * (int)blockDim.x;
    uint4 v[PER];
    uint32_t mx = 0;
    for (int base = 0; base < nv; base += PER * blockDim.x) {
#pragma unroll
        for (int j = 0; j < PER; j++) {
            const int c = base + j * blockDim.x + tid;
            v[j] = c < nv ? __ldg(xv + c) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < PER; j++) {
            const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
            for (int t = 0; t < 4; t++) mx = max(mx, max((w[t] & 0x7FFFu) << 16, w[t] & 0x7FFF0000u));
        }
    }
    for (int o = 16; o; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((tid & 31) == 0) red[tid >> 5] = __uint_as_float(mx);
    __syncthreads();
    if (tid == 0) {
        uint32_t m = 0;
        for (int w = 0; w < (int)(blockDim.x >> 5); w++) m = max(m, __float_as_uint(red[w]));
        red[32] = __uint_as_float((uint32_t)f16_scale_exponent(m));
    }
    __syncthreads();
    const int p = (int)__float_as_uint(red[32]);
    const float s = exp2i(-p);
    for (int base = 0; base < nv; base += PER * blockDim.x) {
        if (!resident) {
#pragma unroll
            for (int j = 0; j < PER; j++) {
                const int c = base + j * blockDim.x + tid;
                v[j] = c < nv ? __ldg(xv + c) : make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int j = 0; j < PER; j++) {
            const int c = base + j * blockDim.x + tid;
            if (c >= nv) continue;
            const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
            uint32_t o[4];
#pragma unroll
            for (int t = 0; t < 4; t++) {
                const __half2 h = __floats2half2_rn(bf16_lo(w[t]) * s, bf16_hi(w[t]) * s);
                o[t] = *reinterpret_cast<const uint32_t*>(&h);
            }
            ov[c] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
    if (tid == 0) *xexp = p;
    __syncthreads();
}

// Row x as three E4M3 terms with per-32 E8M0 block scales (rows 3n, 3n+1, 3n+2 of
// the MX activation buffer): one warp per 32-element block.
__device__ void prep_row_mx(const uint16_t* x, int d, int n, uint8_t* x_mx, uint8_t* x_sc) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    for (int blk = warp; blk < d / 32; blk += nw) {
        const float v = bf16_lo(__ldg(x + blk * 32 + lane));
        uint32_t q[3], sb[3];
        mx3_split(v, q, sb);
#pragma unroll
        for (int t = 0; t < 3; t++) {
            x_mx[(size_t)(3 * n + t) * d + blk * 32 + lane] = (uint8_t)q[t];
            if (lane == 0) x_sc[(size_t)(3 * n + t) * (d / 32) + blk] = (uint8_t)sb[t];
        }
    }
}

__device__ void gemv_slice(const RouteParams& p, int ks, int eg, float* xs /*[N][32][17]*/) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int KS = min(RT_KS, p.d);
    const int k0 = ks * KS;
    const int per_lane = KS / 32;  // 16 (or fewer for small d)
    // the warp's 8 experts are done in two batches of 4; each lane loads its 16 K of
    // a batch up front (the first batch's loads overlap the staging of x)
    const int e0 = eg * RT_EG + warp * 8;
    uint4 wv[4][2];
    auto load_batch = [&](int jb) {
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const int e = e0 + 4 * jb + j;
#pragma unroll
            for (int h = 0; h < 2; h++) {
                wv[j][h] = make_uint4(0, 0, 0, 0);
                if (e < p.E && h * 8 < per_lane) {
                    const uint16_t* src = p.w + (size_t)e * p.d + k0 + lane * per_lane + h * 8;
                    wv[j][h] = __ldg(reinterpret_cast<const uint4*>(src));
                }
            }
        }
    };
    load_batch(0);
    // stage the x slice of every row (fp32) while the weight loads are in flight:
    // row n, lane l's 16 values at xs[(n*32 + l)*17 + c] (padded: conflict-free reads)
    {
        const int nv = p.N * KS / 8;  // 16-byte chunks of the x slice
        for (int base = 0; base < nv; base += 4 * RT_THREADS) {
            uint4 xv[4];
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const int c = base + j * RT_THREADS + tid;
                xv[j] = make_uint4(0, 0, 0, 0);
                if (c < nv) {
                    const int n = c / (KS / 8), off = (c - n * (KS / 8)) * 8;
                    xv[j] = __ldg(reinterpret_cast<const uint4*>(p.x + (size_t)n * p.d + k0 + off));
                }
            }
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const int c = base + j * RT_THREADS + tid;
                if (c >= nv) continue;
                const int n = c / (KS / 8), off = (c - n * (KS / 8)) * 8;
                const uint32_t w[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
#pragma unroll
                for (int t = 0; t < 8; t++) {
                    const int kk = off + t;  // element of the slice
                    const int l = kk / per_lane, cc = kk - l * per_lane;
                    xs[(n * 32 + l) * 17 + cc] = (t & 1) ? bf16_hi(w[t >> 1]) : bf16_lo(w[t >> 1]);
                }
            }
        }
    }
    __syncthreads();
    for (int jb = 0; jb < 2; jb++) {
        if (jb == 1) load_batch(1);
        for (int n = 0; n < p.N; n++) {
            float xr[16];
#pragma unroll
            for (int c = 0; c < 16; c++) xr[c] = (c < per_lane) ? xs[(n * 32 + lane) * 17 + c] : 0.f;
            float s4[4];
#pragma unroll
            for (int j = 0; j < 4; j++) {
                float a = 0.f;
#pragma unroll
                for (int h = 0; h < 2; h++) {
                    const uint32_t q[4] = {wv[j][h].x, wv[j][h].y, wv[j][h].z, wv[j][h].w};
#pragma unroll
                    for (int t = 0; t < 4; t++) {
                        a = fmaf(xr[h * 8 + 2 * t], bf16_lo(q[t]), a);
                        a = fmaf(xr[h * 8 + 2 * t + 1], bf16_hi(q[t]), a);
                    }
                }
                s4[j] = a;
            }
            // transposed butterfly: after 5 levels lane l holds the full sum of
            // expert ((l>>4)&1)*2 + ((l>>3)&1) of the batch
            {
                const bool up = lane & 16;
#pragma unroll
                for (int j = 0; j < 2; j++) {
                    const float send = up ? s4[j] : s4[j + 2];
                    const float keep = up ? s4[j + 2] : s4[j];
                    s4[j] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
                }
            }
            {
                const bool up = lane & 8;
                const float send = up ? s4[0] : s4[1];
                const float keep = up ? s4[1] : s4[0];
                s4[0] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
            }
            s4[0] += __shfl_xor_sync(0xffffffffu, s4[0], 4);
            s4[0] += __shfl_xor_sync(0xffffffffu, s4[0], 2);
            s4[0] += __shfl_xor_sync(0xffffffffu, s4[0], 1);
            if ((lane & 7) == 0) {
                const int j = ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1);
                const int e = e0 + 4 * jb + j;
                if (e < p.E) p.part[((size_t)ks * p.N + n) * p.E + e] = s4[0];
            }
        }
    }
}

// Order-preserving image of a logit: a larger key means a larger value; NaN maps
// below every number and -0 to +0.
__device__ __forceinline__ uint32_t order_key(float v) {
    uint32_t b = __float_as_uint(v);
    b = (b == 0x80000000u) ? 0u : b;
    uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    return isnan(v) ? 0u : ord;
}

__device__ __forceinline__ uint64_t umax64(uint64_t a, uint64_t b) { return a > b ? a : b; }

// largest of 32 keys by a pairwise tree (depth 5)
__device__ __forceinline__ uint64_t tree_max32(const uint64_t (&k)[32]) {
    uint64_t m16[16], m8[8], m4[4];
#pragma unroll
    for (int i = 0; i < 16; i++) m16[i] = umax64(k[2 * i], k[2 * i + 1]);
#pragma unroll
    for (int i = 0; i < 8; i++) m8[i] = umax64(m16[2 * i], m16[2 * i + 1]);
#pragma unroll
    for (int i = 0; i < 4; i++) m4[i] = umax64(m8[2 * i], m8[2 * i + 1]);
    return umax64(umax64(m4[0], m4[1]), umax64(m4[2], m4[3]));
}

__device__ __forceinline__ uint64_t shfl_xor_u64(uint64_t v, int o) {
    const uint32_t lo = __shfl_xor_sync(0xffffffffu, (uint32_t)v, o);
    const uint32_t hi = __shfl_xor_sync(0xffffffffu, (uint32_t)(v >> 32), o);
    return ((uint64_t)hi << 32) | lo;
}

// top-k of one row by one warp.  A candidate's key is (order_key(logit) << 32) |
// (0xFFFFFFFF - expert): the larger key ranks higher (larger logit, then lower
// index, NaN last); 0 means "no candidate".  Lane l holds experts l, l+32, ...;
// each round the warp takes the largest key and the lane that held it rescans.
__device__ void topk_row(const RouteParams& p, const float* lrow, int n, bool from_l2) {
    const int lane = threadIdx.x & 31;
    float v[32];
#pragma unroll
    for (int t = 0; t < 32; t++) {  // every load in flight before any is used
        const int e = min(lane + 32 * t, p.E - 1);
        v[t] = from_l2 ? __ldcg(lrow + e) : lrow[e];
    }
    uint64_t key[32];
    bool any_nan = false;
#pragma unroll
    for (int t = 0; t < 32; t++) {
        const int e = lane + 32 * t;
        const bool ok = e < p.E;
        any_nan |= ok && isnan(v[t]);
        key[t] = ok ? (((uint64_t)order_key(v[t]) << 32) | (uint32_t)(0xFFFFFFFFu - (uint32_t)e)) : 0ull;
    }
    if (__any_sync(0xffffffffu, any_nan) && lane == 0) set_error(p.ctrl, MOE_EBIT_NAN);
    uint64_t local = tree_max32(key);
    uint64_t mine = 0ull;
    for (int j = 0; j < p.k; j++) {
        uint64_t best = local;
#pragma unroll
        for (int o = 16; o; o >>= 1) best = umax64(best, shfl_xor_u64(best, o));
        if (lane == j) mine = best;
        if (best == local) {
#pragma unroll
            for (int t = 0; t < 32; t++) key[t] = (key[t] == best) ? 0ull : key[t];
            local = tree_max32(key);
        }
    }
    const int my_idx = (int)(0xFFFFFFFFu - (uint32_t)mine);
    const float my_val = (lane < p.k) ? (from_l2 ? __ldcg(lrow + my_idx) : lrow[my_idx]) : 0.f;
    // weights: exp(l_j - l_0) / sum_i exp(l_i - l_0), summed in slot order
    const float l0 = __shfl_sync(0xffffffffu, my_val, 0);
    const float ex = (lane < p.k) ? expf(my_val - l0) : 0.f;
    float sum = 0.f;
    for (int j = 0; j < p.k; j++) sum += __shfl_sync(0xffffffffu, ex, j);
    if (lane < p.k) {
        p.topk_idx[(size_t)n * p.k + lane] = my_idx;
        p.topk_w[(size_t)n * p.k + lane] = ex / sum;
    }
}

// Group the block's pairs by expert (N <= 32): smem counts and row bitmaps.
__device__ void group_block(const RouteParams& p, int* s_cnt, uint32_t* s_bits, int* s_off, int* s_idx) {
    const int tid = threadIdx.x;
    const int NK = p.N * p.k;
    for (int e = tid; e < p.E; e += RT_THREADS) {
        s_cnt[e] = 0;
        s_bits[e] = 0;
    }
    __syncthreads();
    for (int i = tid; i < NK; i += RT_THREADS) {
        const int e = __ldcg(p.topk_idx + i);
        s_idx[i] = e;
        if (e >= 0 && e < p.E) {
            atomicAdd(&s_cnt[e], 1);
            atomicOr(&s_bits[e], 1u << (i / p.k));
        }
    }
    __syncthreads();
    // exclusive scan of counts and of the "selected" flags (single warp; E <= 1024)
    if (tid < 32) {
        const int lane = tid;
        const int per = (p.E + 31) / 32;
        const int b = lane * per;
        int c = 0, u = 0;
        for (int e = b; e < min(b + per, p.E); e++) {
            c += s_cnt[e];
            u += s_cnt[e] > 0;
        }
        int cs = c, us = u;
        for (int o = 1; o < 32; o <<= 1) {
            const int a = __shfl_up_sync(0xffffffffu, cs, o);
            const int bb = __shfl_up_sync(0xffffffffu, us, o);
            if (lane >= o) {
                cs += a;
                us += bb;
            }
        }
        cs -= c;
        us -= u;
        for (int e = b; e < min(b + per, p.E); e++) {
            s_off[e] = cs;
            if (s_cnt[e] > 0) {
                p.uexp[us] = e;
                p.off[us] = cs;
                us++;
            }
            cs += s_cnt[e];
        }
        if (lane == 31) {
            p.off[us] = cs;
            p.ctrl[CTRL_UNIQUE] = (uint32_t)us;
            p.ctrl[CTRL_ROWS] = (uint32_t)p.N;
        }
    }
    __syncthreads();
    for (int i = tid; i < NK; i += RT_THREADS) {
        const int e = s_idx[i];
        if (e < 0 || e >= p.E) continue;
        const int n = i / p.k;
        const int rank = __popc(s_bits[e] & ((1u << n) - 1u));
        p.pair[s_off[e] + rank] = i;
    }
    // clean state for the expert kernel
    for (int i = tid; i < p.v_cap; i += RT_THREADS) p.gu_done[i] = 0;
    for (int i = tid; i < p.E; i += RT_THREADS) p.gu_done_tc[i] = 0;
    for (int64_t i = tid; i < p.pairs_cap; i += RT_THREADS) p.hmax[i] = 0;
    if (tid == 0) {
        p.ctrl[CTRL_WORK] = 0;
        p.ctrl[CTRL_EXIT] = 0;
        p.ctrl[CTRL_WORK_TC] = 0;
        p.ctrl[CTRL_EXIT_TC] = 0;
    }
}

__global__ void __launch_bounds__(RT_THREADS, 2) route_kernel(const RouteParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float* smem = reinterpret_cast<float*>(smem_raw);
    __shared__ float red[40];
    __shared__ int s_flag;
    const int tid = threadIdx.x;
    const int b = blockIdx.x;

    if (p.x != nullptr && b < p.N) {
        prep_row(p.x + (size_t)b * p.d, p.d, p.x16 + (size_t)b * p.d, p.xexp + b, red);
        prep_row_mx(p.x + (size_t)b * p.d, p.d, b, p.x_mx, p.x_sc);
    }

    bool group_finisher = false;
    if (b < p.n_gemv_ctas) {
        const int ks = b % p.n_ks, eg = b / p.n_ks;
        gemv_slice(p, ks, eg, smem);
        __threadfence();
        __syncthreads();
        if (tid == 0) s_flag = (atomicAdd(p.ctrl + RT_TICKET_EG + eg, 1u) == (uint32_t)(p.n_ks - 1));
        __syncthreads();
        if (s_flag) {
            __threadfence();
            // sum the K slices in slice order for this group's experts
            const int e_lo = eg * RT_EG, e_hi = min(p.E, e_lo + RT_EG);
            const int span = e_hi - e_lo;
            for (int base = 0; base < p.N * span; base += 4 * RT_THREADS) {
                float v[4][RT_MAX_KS];
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    const int i = base + q * RT_THREADS + tid;
                    const int n = i / span, e = e_lo + (i - n * span);
#pragma unroll
                    for (int ks2 = 0; ks2 < RT_MAX_KS; ks2++)
                        v[q][ks2] = (ks2 < p.n_ks && i < p.N * span)
                                        ? __ldcg(p.part + ((size_t)ks2 * p.N + n) * p.E + e) : 0.f;
                }
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    const int i = base + q * RT_THREADS + tid;
                    if (i >= p.N * span) continue;
                    const int n = i / span, e = e_lo + (i - n * span);
                    float a = 0.f;  // slices summed in slice order
#pragma unroll
                    for (int ks2 = 0; ks2 < RT_MAX_KS; ks2++)
                        if (ks2 < p.n_ks) a += v[q][ks2];
                    p.logits[(size_t)n * p.E + e] = a;
                }
            }
            if (tid == 0) p.ctrl[RT_TICKET_EG + eg] = 0;
            group_finisher = true;
        }
    } else {
        group_finisher = true;  // x-preparation-only CTA (or caller logits)
    }
    if (!group_finisher) return;
    const int participants = (p.n_gemv_ctas > 0 ? p.n_eg : 0) + ((int)gridDim.x - p.n_gemv_ctas);
    __threadfence();
    __syncthreads();
    if (tid == 0) s_flag = (atomicAdd(p.ctrl + CTRL_TICKET, 1u) == (uint32_t)(participants - 1));
    __syncthreads();
    if (!s_flag) return;
    __threadfence();

    // last CTA: selection, weights and grouping for every row
    const int warp = tid >> 5;
    const float* L = p.logits_in ? p.logits_in : p.logits;
    for (int n = warp; n < p.N; n += RT_THREADS / 32) topk_row(p, L + (size_t)n * p.E, n, p.logits_in == nullptr);
    __threadfence();
    __syncthreads();
    int* s_cnt = reinterpret_cast<int*>(smem_raw);
    uint32_t* s_bits = reinterpret_cast<uint32_t*>(s_cnt + 1024);
    int* s_off = reinterpret_cast<int*>(s_bits + 1024);
    int* s_idx = s_off + 1024;
    group_block(p, s_cnt, s_bits, s_off, s_idx);
    if (tid == 0) p.ctrl[CTRL_TICKET] = 0;
}

}  // namespace moe

using namespace moe;

extern "C" int moe_route(const moe_desc* desc, int32_t n_rows, const uint16_t* x, const uint16_t* w_router,
                         const float* logits_in, float* logits_out, int32_t* topk_idx, float* topk_w,
                         void* ws, int32_t n_rows_max, int32_t n_shared, void* stream) {
    if (!desc || !topk_idx || !topk_w || !ws) return MOE_ERR_INVALID_ARG;
    const int d = desc->d_model, f = desc->d_ff, E = desc->n_experts, k = desc->top_k;
    if (desc->group != 32 || d <= 0 || d % 256 || f <= 0 || f % 64 || E <= 0 || E > 1024 || k < 1 ||
        k > 32 || k > E)
        return MOE_ERR_UNSUPPORTED;
    if (n_rows < 1 || n_rows > n_rows_max || n_rows > RT_MAX_ROWS || n_shared < 0) return MOE_ERR_UNSUPPORTED;
    if (!logits_in && (!x || !w_router)) return MOE_ERR_INVALID_ARG;
    if (((uintptr_t)ws & 255) || (x && ((uintptr_t)x & 15)) || (w_router && ((uintptr_t)w_router & 15)))
        return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(d, f, E, k, n_rows_max, n_shared);
    char* base = static_cast<char*>(ws);
    RouteParams p;
    p.d = d;
    p.E = E;
    p.k = k;
    p.N = n_rows;
    p.n_shared = n_shared;
    p.x = x;
    p.w = w_router;
    p.logits_in = logits_in;
    p.logits = logits_out ? logits_out : reinterpret_cast<float*>(base + L.logits);
    p.part = reinterpret_cast<float*>(base + L.h);  // the h buffer is free while routing
    p.topk_idx = topk_idx;
    p.topk_w = topk_w;
    p.ctrl = reinterpret_cast<uint32_t*>(base + L.ctrl);
    p.uexp = reinterpret_cast<int*>(base + L.uexp);
    p.off = reinterpret_cast<int*>(base + L.off);
    p.pair = reinterpret_cast<int*>(base + L.pair);
    p.x16 = reinterpret_cast<__half*>(base + L.x16);
    p.xexp = reinterpret_cast<int*>(base + L.xexp);
    p.gu_done = reinterpret_cast<uint32_t*>(base + L.gu_done);
    p.hmax = reinterpret_cast<uint32_t*>(base + L.hmax);
    p.x_mx = reinterpret_cast<uint8_t*>(base + L.x_mx);
    p.x_sc = reinterpret_cast<uint8_t*>(base + L.x_sc);
    p.gu_done_tc = reinterpret_cast<uint32_t*>(base + L.gu_done_tc);
    p.v_cap = n_shared + (n_rows_max * k < E ? n_rows_max * k : E);
    p.pairs_cap = L.pairs;
    const int KS = d < RT_KS ? d : RT_KS;
    p.n_ks = d / KS;
    p.n_eg = (E + RT_EG - 1) / RT_EG;
    if (p.n_eg > 32 || p.n_ks > RT_MAX_KS) return MOE_ERR_UNSUPPORTED;
    // the partial logits must fit in the h buffer: n_ks * N * E floats
    if ((size_t)p.n_ks * n_rows * E * 4 > L.dbg_g - L.h) return MOE_ERR_UNSUPPORTED;
    p.n_gemv_ctas = logits_in ? 0 : p.n_ks * p.n_eg;
    int grid = p.n_gemv_ctas > n_rows ? p.n_gemv_ctas : n_rows;
    const size_t smem = (size_t)RT_MAX_ROWS * 32 * 17 * 4;  // padded x slice (also covers the grouping tables)
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return MOE_ERR_CUDA;
        attr_set = true;
    }
    route_kernel<<<grid, RT_THREADS, smem, static_cast<cudaStream_t>(stream)>>>(p);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
