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
static_assert(RT_THREADS == 256, "topk_row_cta: one histogram bin and 4 experts per thread");
constexpr int RT_KS = 512;      // K elements per slice
constexpr int RT_EG = 64;       // experts per group (8 per warp)
constexpr int RT_MAX_ROWS = 32;
constexpr int RT_MAX_KS = 16;   // K slices: d <= 8192
constexpr int RT_TICKET_EG = 32;  // ctrl words [32, 64) hold the per-group tickets
constexpr int RT_CAND_ROWS = 4;   // router-GEMV blocks of up to this many rows merge per-group candidates

struct RouteParams {
    int d, E, k, N, n_shared;
    int n_ks, n_eg, n_gemv_ctas;
    const uint16_t* x;
    const uint16_t* w;
    const float* logits_in;
    float* logits;        // logits_out, or the workspace copy
    float* part;          // [n_ks][N][E] partial logits
    uint64_t* cand;       // [N][n_eg][k] per-group top-k candidates (selection key << 32 | ~expert), ranked
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
    uint8_t* x_mx;        // [MX_TERMS N][d/2] packed E2M1 terms of x for the block-scaled expert kernel
    uint8_t* x_sc;        // [MX_TERMS N][d/32] their E8M0 scales
    uint32_t* gu_done_tc;
    uint32_t* rbits;      // blocks of more than 32 rows: [groups][E] row bitmaps
    uint32_t* rbits2;
    int* rbase;
    int v_cap;
    int64_t pairs_cap;
};

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// E2M1 split of one 1024-element chunk of row n (four blocks per warp, loads
// first), and the chunk's max |x| published for the row's f16 copy
constexpr int RT_CHUNK = 1024;
__device__ void prep_chunk_mx(const RouteParams& p, int n, int c) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nblk = p.d / 32;
    const uint16_t* x = p.x + (size_t)n * p.d;
    float v[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int blk = c * (RT_CHUNK / 32) + warp * 4 + i;
        v[i] = blk < nblk ? bf16_lo(__ldg(x + blk * 32 + lane)) : 0.f;
    }
    uint32_t mx = 0;
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int blk = c * (RT_CHUNK / 32) + warp * 4 + i;
        if (blk >= nblk) continue;
        mx = max(mx, __float_as_uint(v[i]) & 0x7FFFFFFFu);
        uint32_t q[MX_TERMS], sb[MX_TERMS];
        mx_split(v[i], q, sb);
#pragma unroll
        for (int t = 0; t < MX_TERMS; t++) {
            store_e2m1_block(p.x_mx + (size_t)(MX_TERMS * n + t) * (p.d / 2) + blk * 16, q[t]);
            if (lane == 0) p.x_sc[(size_t)(MX_TERMS * n + t) * nblk + blk] = (uint8_t)sb[t];
        }
    }
    mx = __reduce_max_sync(0xffffffffu, mx);
    if (lane == 0 && mx != 0u && n < RT_MAX_ROWS) atomicMax(p.ctrl + CTRL_XMAX + n, mx);
}

// Activation preparation for the f16 (shared-expert) path: x16 = f16(x * 2^-p),
// p chosen from the row's largest magnitude (published by the CTAs that read the
// row) so the row sits inside the f16 range; vectorised, all loads of a pass first.
__device__ void prep_row_x16(const uint16_t* x, int d, uint32_t maxbits, __half* x16, int* xexp) {
    const int p = f16_scale_exponent(maxbits);
    const float s = exp2i(-p);
    const uint4* xv = reinterpret_cast<const uint4*>(x);
    uint4* ov = reinterpret_cast<uint4*>(x16);
    const int nv = d / 8;
    for (int base = 0; base < nv; base += 4 * blockDim.x) {
        uint4 v[4];
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const int c = base + j * blockDim.x + threadIdx.x;
            v[j] = c < nv ? __ldg(xv + c) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const int c = base + j * blockDim.x + threadIdx.x;
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
    if (threadIdx.x == 0) *xexp = p;
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
    // publish each row's max |x| over this slice, and split the slice's 32-element
    // blocks of rows n = eg (mod n_eg) into E2M1 terms (all from the staged copy)
    for (int n = warp; n < p.N; n += RT_THREADS / 32) {
        uint32_t mx = 0;
        for (int c = 0; c < per_lane; c++) mx = max(mx, __float_as_uint(xs[(n * 32 + lane) * 17 + c]) & 0x7FFFFFFFu);
        for (int o = 16; o; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 0) atomicMax(p.ctrl + CTRL_XMAX + n, mx);
    }
    {
        const int nblk = KS / 32;
        int task = warp;
        for (int n = eg; n < p.N; n += p.n_eg) {
            for (; task < nblk; task += RT_THREADS / 32) {
                const int el = task * 32 + lane;  // element of the slice
                const float v = xs[(n * 32 + el / per_lane) * 17 + el % per_lane];
                uint32_t q[MX_TERMS], sb[MX_TERMS];
                mx_split(v, q, sb);
                const int blk = (k0 >> 5) + task;
#pragma unroll
                for (int t = 0; t < MX_TERMS; t++) {
                    store_e2m1_block(p.x_mx + (size_t)(MX_TERMS * n + t) * (p.d / 2) + (k0 + task * 32) / 2, q[t]);
                    if (lane == 0) p.x_sc[(size_t)(MX_TERMS * n + t) * (p.d / 32) + blk] = (uint8_t)sb[t];
                }
            }
            task -= nblk;
        }
    }
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
// Selection key of a logit: larger ranks higher, +0 and -0 equal, NaN (1) below
// every number, 0 = no candidate.
__device__ __forceinline__ uint32_t sel_key(float v) {
    uint32_t b = __float_as_uint(v);
    b = (b == 0x80000000u) ? 0u : b;
    const uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    return isnan(v) ? 1u : ord;
}

// the logit a key came from (-0 comes back as +0)
__device__ __forceinline__ float key_value(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// expert held by key t of `lane` (t = 4 i + j): e = 128 i + 4 lane + j when the
// row was read as float4 (E % 4 == 0), else e = lane + 32 t; either way a lane's
// experts increase with t
__device__ __forceinline__ int key_expert(int t, int lane, bool vec) {
    return vec ? 128 * (t >> 2) + 4 * lane + (t & 3) : lane + 32 * t;
}

// top-k of one row by one warp, with ties going to the lower index.  Every load
// is issued before any is used.  The k-th largest key T is found bit by bit
// (most significant first) from warp-wide counts of the keys >= a candidate,
// stopping as soon as exactly k keys qualify; keys above T are all taken and the
// keys equal to T are taken in index order.  The k winners are then ranked
// (larger key first, then lower index) through shared memory `sel` (2k words).
// If `sidx` is given, the selected experts also go there (shared memory, k words).
__device__ void topk_row(const RouteParams& p, const float* lrow, int n, bool from_l2, uint32_t* sel, int* sidx) {
    const int lane = threadIdx.x & 31, K = p.k;
    const bool vec = (p.E & 3) == 0 && ((uintptr_t)lrow & 15) == 0;
    uint32_t key[32];
    if (vec) {
        float4 v[8];
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const int e0 = 128 * i + 4 * lane;
            v[i] = e0 < p.E ? (from_l2 ? __ldcg(reinterpret_cast<const float4*>(lrow + e0))
                                       : __ldg(reinterpret_cast<const float4*>(lrow + e0)))
                            : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const bool ok = 128 * i + 4 * lane < p.E;
            key[4 * i + 0] = ok ? sel_key(v[i].x) : 0u;
            key[4 * i + 1] = ok ? sel_key(v[i].y) : 0u;
            key[4 * i + 2] = ok ? sel_key(v[i].z) : 0u;
            key[4 * i + 3] = ok ? sel_key(v[i].w) : 0u;
        }
    } else {
        float v[32];
#pragma unroll
        for (int t = 0; t < 32; t++) {
            const int e = lane + 32 * t;
            v[t] = e < p.E ? (from_l2 ? __ldcg(lrow + e) : __ldg(lrow + e)) : 0.f;
        }
#pragma unroll
        for (int t = 0; t < 32; t++) key[t] = lane + 32 * t < p.E ? sel_key(v[t]) : 0u;
    }
    bool any_nan = false;
#pragma unroll
    for (int t = 0; t < 32; t++) any_nan |= key[t] == 1u;
    if (__any_sync(0xffffffffu, any_nan) && lane == 0) set_error(p.ctrl, MOE_EBIT_NAN);

    // T: the largest value with at least K keys >= T
    uint32_t T = 0u;
    for (int bit = 31; bit >= 0; bit--) {
        const uint32_t cand = T | (1u << bit);
        uint32_t c = 0;
#pragma unroll
        for (int t = 0; t < 32; t++) c += key[t] >= cand ? 1u : 0u;
        c = __reduce_add_sync(0xffffffffu, c);
        if (c >= (uint32_t)K) T = cand;
        if (c == (uint32_t)K) break;  // exactly K keys are >= cand: they are the top K
    }
    uint32_t n_gt = 0, n_ge = 0;
#pragma unroll
    for (int t = 0; t < 32; t++) {
        n_gt += key[t] > T ? 1u : 0u;
        n_ge += key[t] >= T ? 1u : 0u;
    }
    n_gt = __reduce_add_sync(0xffffffffu, n_gt);
    n_ge = __reduce_add_sync(0xffffffffu, n_ge);
    uint32_t take_eq = 0xFFFFFFFFu;  // bit t: key t equal to T is taken
    if (n_ge > (uint32_t)K) {
        // ties at T: take them in index order until K are selected
        int need = K - (int)n_gt;
        take_eq = 0u;
        // index order: blocks i, then lanes, then j (vec: experts 128 i + 4 lane + j);
        // t, then lanes otherwise
        if (vec) {
#pragma unroll
            for (int i = 0; i < 8; i++) {
                if (need <= 0) break;
                uint32_t cnt = 0;
#pragma unroll
                for (int j = 0; j < 4; j++) cnt += key[4 * i + j] == T ? 1u : 0u;
                // lanes below this one hold lower indices in block i
                uint32_t before = cnt;
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t up = __shfl_up_sync(0xffffffffu, before, o);
                    if (lane >= o) before += up;
                }
                before -= cnt;  // exclusive
                const uint32_t tot = __shfl_sync(0xffffffffu, before + cnt, 31);
                int mine = need - (int)before;  // how many of this lane's ties in block i are taken
#pragma unroll
                for (int j = 0; j < 4; j++) {
                    if (key[4 * i + j] == T && mine > 0) {
                        take_eq |= 1u << (4 * i + j);
                        mine--;
                    }
                }
                need -= (int)min(tot, (uint32_t)max(need, 0));
            }
        } else {
#pragma unroll
            for (int t = 0; t < 32; t++) {
                if (need <= 0) break;
                const uint32_t bal = __ballot_sync(0xffffffffu, key[t] == T);
                const uint32_t before = __popc(bal & ((1u << lane) - 1u));
                if (key[t] == T && (int)before < need) take_eq |= 1u << t;
                need -= min(__popc(bal), need);
            }
        }
    }
    // compact the K winners (order irrelevant here), then rank them
    uint32_t mine = 0;
#pragma unroll
    for (int t = 0; t < 32; t++) mine += (key[t] > T || (key[t] == T && (take_eq >> t) & 1u)) ? 1u : 0u;
    uint32_t at = mine;
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t up = __shfl_up_sync(0xffffffffu, at, o);
        if (lane >= o) at += up;
    }
    at -= mine;
#pragma unroll
    for (int t = 0; t < 32; t++) {
        if (key[t] > T || (key[t] == T && (take_eq >> t) & 1u)) {
            sel[at] = key[t];
            sel[K + at] = (uint32_t)key_expert(t, lane, vec);
            at++;
        }
    }
    __syncwarp();
    uint32_t wk = 0u, wi = 0u;
    int rank = 0;
    if (lane < K) {
        wk = sel[lane];
        wi = sel[K + lane];
        for (int j = 0; j < K; j++) {
            const uint32_t kj = sel[j], ij = sel[K + j];
            rank += (kj > wk || (kj == wk && ij < wi)) ? 1 : 0;
        }
    }
    __syncwarp();
    if (lane < K) {
        sel[rank] = wk;
        sel[K + rank] = wi;
    }
    __syncwarp();
    const uint32_t my_key = lane < K ? sel[lane] : 0u;
    const int my_idx = lane < K ? (int)sel[K + lane] : 0;
    __syncwarp();
    const float my_val = (lane < K) ? key_value(my_key) : 0.f;
    // weights: exp(l_j - l_0) / sum_i exp(l_i - l_0), summed in slot order
    const float l0 = __shfl_sync(0xffffffffu, my_val, 0);
    const float ex = (lane < K) ? expf(my_val - l0) : 0.f;
    float sum = 0.f;
    for (int j = 0; j < K; j++) sum += __shfl_sync(0xffffffffu, ex, j);
    if (lane < K) {
        p.topk_idx[(size_t)n * K + lane] = my_idx;
        p.topk_w[(size_t)n * K + lane] = ex / sum;
        if (sidx) sidx[lane] = my_idx;
    }
}

// top-k of one row by the whole CTA (RT_THREADS threads; blocks of one or two
// rows, where one warp per row would leave the CTA idle): thread t holds the
// keys of experts 4t..4t+3.  The k-th largest key T is found by radix selection,
// 8 bits per round from the most significant, with a shared-memory histogram per
// round; keys above T are all taken and keys equal to T in index order (a block
// scan of the tie counts); the k winners are ranked as in topk_row.  Same
// selection and weight arithmetic as topk_row.  `s` is 2 KB of shared memory.
__device__ void topk_row_cta(const RouteParams& p, const float* lrow, int n, bool from_l2, uint32_t* s, int* sidx) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, K = p.k, E = p.E;
    uint32_t* hist = s;                         // [256]
    uint32_t* wsum = s + 256;                   // [8] per-warp totals, [8] second scan
    uint32_t* bc = s + 272;                     // [4] broadcast: prefix, remaining k, ...
    uint32_t* sel = s + 288;                    // [2k]
    uint32_t key[4];
    const int e0 = 4 * tid;
    bool nan = false;
    if ((E & 3) == 0 && ((uintptr_t)lrow & 15) == 0) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (e0 < E)
            v = from_l2 ? __ldcg(reinterpret_cast<const float4*>(lrow + e0))
                        : __ldg(reinterpret_cast<const float4*>(lrow + e0));
        const float f[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; j++) {
            key[j] = e0 + j < E ? sel_key(f[j]) : 0u;
            nan |= e0 + j < E && isnan(f[j]);
        }
    } else {
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const float f = e0 + j < E ? (from_l2 ? __ldcg(lrow + e0 + j) : __ldg(lrow + e0 + j)) : 0.f;
            key[j] = e0 + j < E ? sel_key(f) : 0u;
            nan |= e0 + j < E && isnan(f);
        }
    }
    if (__syncthreads_or(nan) && tid == 0) set_error(p.ctrl, MOE_EBIT_NAN);

    // radix selection: after round r, prefix holds the top 8(r+1) bits of T and
    // rem the number of keys equal to T on those bits still to take
    uint32_t prefix = 0u, rem = (uint32_t)K;
    for (int r = 0; r < 4; r++) {
        const int shift = 24 - 8 * r;
        hist[tid] = 0u;  // RT_THREADS == 256 bins
        __syncthreads();
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const bool match = r == 0 || (key[j] >> (shift + 8)) == (prefix >> (shift + 8));
            if (match && key[j] != 0u) atomicAdd(&hist[(key[j] >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (warp == 0) {
            // lane l holds bins 255-8l .. 248-8l (descending); counts above each bin
            uint32_t c[8], tot = 0;
#pragma unroll
            for (int j = 0; j < 8; j++) {
                c[j] = hist[255 - 8 * lane - j];
                tot += c[j];
            }
            uint32_t incl = tot;
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t up = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += up;
            }
            uint32_t above = incl - tot;  // keys in higher bins than this lane's first
            int hit = -1;
            uint32_t hit_above = 0;
#pragma unroll
            for (int j = 0; j < 8; j++) {
                if (hit < 0 && above < rem && above + c[j] >= rem) {
                    hit = j;
                    hit_above = above;
                }
                above += c[j];
            }
            const uint32_t m = __ballot_sync(0xffffffffu, hit >= 0);
            const int src = __ffs(m) - 1;  // exactly one lane holds the bin
            const int hb = __shfl_sync(0xffffffffu, hit, src);
            const uint32_t ha = __shfl_sync(0xffffffffu, hit_above, src);
            if (lane == 0) {
                bc[0] = prefix | ((uint32_t)(255 - 8 * src - hb) << shift);
                bc[1] = rem - ha;
            }
        }
        __syncthreads();
        prefix = bc[0];
        rem = bc[1];
    }
    const uint32_t T = prefix;
    // rem keys equal to T are taken, in index order; every key above T is taken
    uint32_t n_take = 0, n_tie = 0;
#pragma unroll
    for (int j = 0; j < 4; j++) {
        n_take += key[j] > T ? 1u : 0u;
        n_tie += key[j] == T ? 1u : 0u;
    }
    // exclusive block scans of the tie counts and of the takes (thread order = index order)
    uint32_t it = n_tie, ik = n_take;
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t a = __shfl_up_sync(0xffffffffu, it, o), b = __shfl_up_sync(0xffffffffu, ik, o);
        if (lane >= o) {
            it += a;
            ik += b;
        }
    }
    if (lane == 31) {
        wsum[warp] = it;
        wsum[8 + warp] = ik;
    }
    __syncthreads();
    uint32_t tie_before = it - n_tie, take_before = ik - n_take;
    for (int w = 0; w < warp; w++) {
        tie_before += wsum[w];
        take_before += wsum[8 + w];
    }
    // ties taken by the threads before this one: min(tie_before, rem)
    uint32_t at = take_before + min(tie_before, rem);
    uint32_t ties_left = tie_before < rem ? rem - tie_before : 0u;
#pragma unroll
    for (int j = 0; j < 4; j++) {
        const bool take = key[j] > T || (key[j] == T && ties_left > 0u);
        if (key[j] == T && ties_left > 0u) ties_left--;
        if (take) {
            sel[at] = key[j];
            sel[K + at] = (uint32_t)(e0 + j);
            at++;
        }
    }
    __syncthreads();
    if (warp == 0) {
        uint32_t wk = 0u, wi = 0u;
        int rank = 0;
        if (lane < K) {
            wk = sel[lane];
            wi = sel[K + lane];
            for (int j = 0; j < K; j++) {
                const uint32_t kj = sel[j], ij = sel[K + j];
                rank += (kj > wk || (kj == wk && ij < wi)) ? 1 : 0;
            }
        }
        __syncwarp();
        if (lane < K) {
            sel[rank] = wk;
            sel[K + rank] = wi;
        }
        __syncwarp();
        const uint32_t my_key = lane < K ? sel[lane] : 0u;
        const int my_idx = lane < K ? (int)sel[K + lane] : 0;
        const float my_val = (lane < K) ? key_value(my_key) : 0.f;
        // weights: exp(l_j - l_0) / sum_i exp(l_i - l_0), summed in slot order
        const float l0 = __shfl_sync(0xffffffffu, my_val, 0);
        const float ex = (lane < K) ? expf(my_val - l0) : 0.f;
        float sum = 0.f;
        for (int j = 0; j < K; j++) sum += __shfl_sync(0xffffffffu, ex, j);
        if (lane < K) {
            p.topk_idx[(size_t)n * K + lane] = my_idx;
            p.topk_w[(size_t)n * K + lane] = ex / sum;
            if (sidx) sidx[lane] = my_idx;
        }
    }
    __syncthreads();  // s is reused by the next row
}

// Selection order of a row's experts as one 64-bit key: the logit's selection key
// above the complemented expert index, so equal logits rank by lower index and no
// two experts of a row compare equal (0 = no candidate).
__device__ __forceinline__ uint64_t cand_key(float v, int e) {
    return ((uint64_t)sel_key(v) << 32) | (uint64_t)(~(uint32_t)e);
}

// A group finisher of a router-GEMV block of up to RT_CAND_ROWS rows: the k best of
// its experts e_lo .. e_lo + span - 1 in every row (logits in s_lg[n][RT_EG]),
// ranked, into p.cand.  One thread per (row, expert) counts the group's experts
// that rank above it; ranks the group cannot fill (span < k) get no candidate.
__device__ void group_candidates(const RouteParams& p, int eg, int span, const float* s_lg, uint64_t* s_ck) {
    const int tid = threadIdx.x, K = p.k;
    const int total = p.N * RT_EG;
    bool nan = false;
    for (int i = tid; i < total; i += RT_THREADS) {
        const int j = i % RT_EG;
        uint64_t c = 0;
        if (j < span) {
            const float v = s_lg[i];
            nan |= isnan(v);
            c = cand_key(v, eg * RT_EG + j);
        }
        s_ck[i] = c;
    }
    if (__syncthreads_or(nan) && tid == 0) set_error(p.ctrl, MOE_EBIT_NAN);
    for (int i = tid; i < total; i += RT_THREADS) {
        const int n = i / RT_EG, j = i - n * RT_EG;
        if (j >= span) continue;
        const uint64_t mine = s_ck[i];
        const uint64_t* row = s_ck + n * RT_EG;
        int rank = 0;
#pragma unroll 8
        for (int t = 0; t < RT_EG; t++) rank += row[t] > mine ? 1 : 0;
        if (rank < K) p.cand[((size_t)n * p.n_eg + eg) * K + rank] = mine;
    }
    for (int i = tid; i < p.N * K; i += RT_THREADS) {
        const int n = i / K, r = i - n * K;
        if (r >= span) p.cand[((size_t)n * p.n_eg + eg) * K + r] = 0;
    }
}

// The last CTA of a router-GEMV block of up to RT_CAND_ROWS rows: every row's k
// winners from the groups' ranked candidates.  A candidate's rank in the row is
// its rank in its own group plus, for every other group, the number of that
// group's candidates above it (a binary search in the group's descending list).
// The winners are then weighted by a warp per row with the arithmetic of topk_row.
// s_c: [N][n_eg k] candidates, s_sel: [N][k] winners (shared memory).
__device__ void select_from_candidates(const RouteParams& p, uint64_t* s_c, uint64_t* s_sel, int* sidx) {
    const int tid = threadIdx.x, K = p.k, G = p.n_eg, M = G * K;
    const int total = p.N * M;
    for (int i = tid; i < total; i += RT_THREADS) s_c[i] = __ldcg(p.cand + i);
    __syncthreads();
    for (int i = tid; i < total; i += RT_THREADS) {
        const int n = i / M, rest = i - n * M, g = rest / K, r = rest - g * K;
        const uint64_t mine = s_c[i];
        if (mine == 0) continue;
        const uint64_t* rowc = s_c + n * M;
        int rank = r;
        for (int g2 = 0; g2 < G && rank < K; g2++) {
            if (g2 == g) continue;
            const uint64_t* l = rowc + g2 * K;
            int lo = 0, hi = K;  // the first entry of list g2 that is not above `mine`
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (l[mid] > mine) lo = mid + 1;
                else hi = mid;
            }
            rank += lo;
        }
        if (rank < K) s_sel[n * K + rank] = mine;
    }
    __syncthreads();
    const int lane = tid & 31, warp = tid >> 5;
    for (int n = warp; n < p.N; n += RT_THREADS / 32) {
        const uint64_t c = lane < K ? s_sel[n * K + lane] : 0;
        const uint32_t my_key = (uint32_t)(c >> 32);
        const int my_idx = (int)~(uint32_t)c;
        const float my_val = (lane < K) ? key_value(my_key) : 0.f;
        // weights: exp(l_j - l_0) / sum_i exp(l_i - l_0), summed in slot order
        const float l0 = __shfl_sync(0xffffffffu, my_val, 0);
        const float ex = (lane < K) ? expf(my_val - l0) : 0.f;
        float sum = 0.f;
        for (int j = 0; j < K; j++) sum += __shfl_sync(0xffffffffu, ex, j);
        if (lane < K) {
            p.topk_idx[(size_t)n * K + lane] = my_idx;
            p.topk_w[(size_t)n * K + lane] = ex / sum;
            sidx[n * K + lane] = my_idx;
        }
    }
}

// the expert kernels' counters and maxima, cleared by the routing for its block
__device__ void reset_expert_state(const RouteParams& p) {
    const int tid = threadIdx.x;
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

// Group a block of N k <= RT_THREADS pairs by expert (s_idx: the selections, pair
// i = row * k + slot): pair i's place among the pairs sorted by (expert, i) is the
// number of pairs before it in that order, and an expert's place among the
// selected experts the number of distinct experts below it (counted over the
// first pair of each).  The same order as group_block.
__device__ void group_small(const RouteParams& p, const int* s_idx, int* s_first) {
    const int tid = threadIdx.x, NK = p.N * p.k;
    int e = 0, pos = 0;
    bool first = false, valid = false;
    if (tid < NK) {
        e = s_idx[tid];
        valid = e >= 0 && e < p.E;
        first = valid;
        for (int j = 0; j < NK; j++) {
            const int ej = s_idx[j];
            const bool vj = ej >= 0 && ej < p.E;
            pos += (vj && (ej < e || (ej == e && j < tid))) ? 1 : 0;
            if (ej == e && j < tid) first = false;
        }
        s_first[tid] = first ? e : INT_MAX;
    }
    __syncthreads();
    if (valid) {
        int u = 0;
        for (int j = 0; j < NK; j++) u += s_first[j] < e ? 1 : 0;
        p.pair[pos] = tid;
        if (first) {
            p.uexp[u] = e;
            p.off[u] = pos;
        }
    }
    if (tid == 0) {
        int U = 0, total = 0;
        for (int j = 0; j < NK; j++) {
            U += s_first[j] != INT_MAX ? 1 : 0;
            total += (s_idx[j] >= 0 && s_idx[j] < p.E) ? 1 : 0;
        }
        p.off[U] = total;
        p.ctrl[CTRL_UNIQUE] = (uint32_t)U;
        p.ctrl[CTRL_ROWS] = (uint32_t)p.N;
    }
    reset_expert_state(p);
}

// Group the block's pairs by expert (N <= 32): smem counts and row bitmaps; s_idx
// holds the block's selections (N k words, written by topk_row).
__device__ void group_block(const RouteParams& p, int* s_cnt, uint32_t* s_bits, int* s_off, int* s_idx) {
    const int tid = threadIdx.x;
    const int NK = p.N * p.k;
    for (int e = tid; e < p.E; e += RT_THREADS) {
        s_cnt[e] = 0;
        s_bits[e] = 0;
    }
    __syncthreads();
    for (int i = tid; i < NK; i += RT_THREADS) {
        const int e = s_idx[i];
        if (e >= 0 && e < p.E) {
            atomicAdd(&s_cnt[e], 1);
            atomicOr(&s_bits[e], 1u << (i / p.k));
        }
    }
    __syncthreads();
    // exclusive scans over the experts of the counts and of the "selected" flags:
    // thread t holds experts 4t..4t+3 (E <= 1024 = 4 RT_THREADS)
    __shared__ int s_wc[RT_THREADS / 32], s_wu[RT_THREADS / 32];
    {
        const int lane = tid & 31, warp = tid >> 5;
        int c[4], ct = 0, ut = 0;
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const int e = 4 * tid + j;
            c[j] = e < p.E ? s_cnt[e] : 0;
            ct += c[j];
            ut += c[j] > 0 ? 1 : 0;
        }
        int ic = ct, iu = ut;
        for (int o = 1; o < 32; o <<= 1) {
            const int a = __shfl_up_sync(0xffffffffu, ic, o), bu = __shfl_up_sync(0xffffffffu, iu, o);
            if (lane >= o) {
                ic += a;
                iu += bu;
            }
        }
        if (lane == 31) {
            s_wc[warp] = ic;
            s_wu[warp] = iu;
        }
        __syncthreads();
        int cs = ic - ct, us = iu - ut, c_all = 0, u_all = 0;
        for (int w = 0; w < RT_THREADS / 32; w++) {
            if (w < warp) {
                cs += s_wc[w];
                us += s_wu[w];
            }
            c_all += s_wc[w];
            u_all += s_wu[w];
        }
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const int e = 4 * tid + j;
            if (e >= p.E) break;
            s_off[e] = cs;
            if (c[j] > 0) {
                p.uexp[us] = e;
                p.off[us] = cs;
                us++;
            }
            cs += c[j];
        }
        if (tid == 0) {
            p.off[u_all] = c_all;
            p.ctrl[CTRL_UNIQUE] = (uint32_t)u_all;
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
    reset_expert_state(p);
}

__global__ void __launch_bounds__(RT_THREADS, 2) route_kernel(const RouteParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float* smem = reinterpret_cast<float*>(smem_raw);
    __shared__ int s_flag;
    const int tid = threadIdx.x;
    const int b = blockIdx.x;
    // the shared experts of the block may start beside the routing (they need x only)
    griddep_launch_dependents();
    const bool stamp = tid == 0 && p.n_gemv_ctas > 0;  // timeline of the router-GEMV launch
    if (stamp) tl_begin(p.ctrl, TL_ROUTE);

    if (p.x != nullptr && p.n_gemv_ctas == 0) {  // caller logits: one CTA per (row, chunk)
        const int nc = (p.d + RT_CHUNK - 1) / RT_CHUNK;
        const int n = b / nc, c = b - n * nc;
        prep_chunk_mx(p, n, c);
        // the row's last chunk writes its f16 copy
        __threadfence();
        __syncthreads();
        if (tid == 0) s_flag = (atomicAdd(p.ctrl + RT_TICKET_EG + n, 1u) == (uint32_t)(nc - 1));
        __syncthreads();
        if (s_flag) {
            __threadfence();
            prep_row_x16(p.x + (size_t)n * p.d, p.d, __ldcg(p.ctrl + CTRL_XMAX + n), p.x16 + (size_t)n * p.d,
                         p.xexp + n);
            if (tid == 0) p.ctrl[RT_TICKET_EG + n] = 0;
        }
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
            // sum the K slices in slice order for this group's experts (small blocks
            // also keep them in shared memory for the group's candidates)
            const int e_lo = eg * RT_EG, e_hi = min(p.E, e_lo + RT_EG);
            const int span = e_hi - e_lo;
            const bool cand = p.N <= RT_CAND_ROWS;
            float* s_lg = smem;                                            // [N][RT_EG]
            uint64_t* s_ck = reinterpret_cast<uint64_t*>(smem_raw + 4096);  // [N][RT_EG]
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
                    if (cand) s_lg[n * RT_EG + (e - e_lo)] = a;
                }
            }
            if (cand) {
                __syncthreads();
                group_candidates(p, eg, span, s_lg, s_ck);
            }
            if (tid == 0) p.ctrl[RT_TICKET_EG + eg] = 0;
            group_finisher = true;
        }
    } else {
        group_finisher = true;  // x-preparation-only CTA (or caller logits)
    }
    if (!group_finisher) {
        if (stamp) tl_end(p.ctrl, TL_ROUTE);
        return;
    }
    const bool gemv_finisher = b < p.n_gemv_ctas;
    const int participants = (p.n_gemv_ctas > 0 ? p.n_eg : 0) + ((int)gridDim.x - p.n_gemv_ctas);
    __threadfence();
    __syncthreads();
    if (tid == 0) s_flag = (atomicAdd(p.ctrl + CTRL_TICKET, 1u) == (uint32_t)(participants - 1));
    __syncthreads();
    const bool last = s_flag != 0;
    if (last) {
        __threadfence();
        // last CTA: selection, weights and grouping for every row (tables in shared
        // memory: grouping [0, 16 KB), selections [32 KB, 34 KB))
        const int warp = tid >> 5;
        const float* L = p.logits_in ? p.logits_in : p.logits;
        int* s_cnt = reinterpret_cast<int*>(smem_raw);
        uint32_t* s_bits = reinterpret_cast<uint32_t*>(s_cnt + 1024);
        int* s_off = reinterpret_cast<int*>(s_bits + 1024);
        int* s_idx = s_off + 1024;
        if (p.n_gemv_ctas > 0 && p.N <= RT_CAND_ROWS) {  // merge the groups' candidates
            select_from_candidates(p, reinterpret_cast<uint64_t*>(smem_raw + 16384),
                                   reinterpret_cast<uint64_t*>(smem_raw + 32768), s_idx);
        } else if (p.N <= 2) {  // the whole CTA on each row
            uint32_t* s_topk = reinterpret_cast<uint32_t*>(smem_raw + 32768);
            for (int n = 0; n < p.N; n++)
                topk_row_cta(p, L + (size_t)n * p.E, n, p.logits_in == nullptr, s_topk, s_idx + n * p.k);
        } else {  // a warp per row
            uint32_t* sel = reinterpret_cast<uint32_t*>(smem_raw + 32768) + warp * 64;  // 2k words per warp
            for (int n = warp; n < p.N; n += RT_THREADS / 32)
                topk_row(p, L + (size_t)n * p.E, n, p.logits_in == nullptr, sel, s_idx + n * p.k);
        }
        __syncthreads();
        if (p.N * p.k <= RT_THREADS)
            group_small(p, s_idx, s_cnt);
        else
            group_block(p, s_cnt, s_bits, s_off, s_idx);
        if (tid == 0) p.ctrl[CTRL_TICKET] = 0;
        if (stamp) tl_end(p.ctrl, TL_ROUTE);  // the routing is complete
        if (!gemv_finisher) {  // caller logits: every row's f16 copy is already written
            for (int n = tid; n < RT_MAX_ROWS; n += RT_THREADS) p.ctrl[CTRL_XMAX + n] = 0;
            return;
        }
    }
    if (!gemv_finisher) return;
    // every CTA has published every row's max: the finisher of group eg writes the
    // f16 copies of rows n = eg (mod n_eg), after the selection (nothing in this
    // launch waits for them); the last finisher to get here clears the maxima
    const int eg = b / p.n_ks;
    for (int n = eg; n < p.N; n += p.n_eg)
        prep_row_x16(p.x + (size_t)n * p.d, p.d, __ldcg(p.ctrl + CTRL_XMAX + n), p.x16 + (size_t)n * p.d,
                     p.xexp + n);
    __syncthreads();
    if (tid == 0 && atomicAdd(p.ctrl + CTRL_RT_DONE, 1u) == (uint32_t)(p.n_eg - 1)) {
        for (int n = 0; n < RT_MAX_ROWS; n++) p.ctrl[CTRL_XMAX + n] = 0;
        p.ctrl[CTRL_RT_DONE] = 0;
    }
    if (stamp) tl_end(p.ctrl, TL_ROUTE);
}

// ---------------------------------------------------------------------------
// blocks of more than 32 rows (prefill), caller logits: three launches
// ---------------------------------------------------------------------------

// per row (one warp each): the top-k and its weights, and the row's bit in the
// bitmap of every expert it selected (its 32-row group); the other CTAs split the
// rows into E2M1 terms for the expert kernel
__global__ void __launch_bounds__(RT_THREADS) route_rows_kernel(const RouteParams p, int n_topk_ctas) {
    __shared__ uint32_t sel[RT_THREADS / 32][64];
    const int b = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (b < n_topk_ctas) {
        const int n = b * (RT_THREADS / 32) + warp;
        if (n >= p.N) return;
        topk_row(p, p.logits_in + (size_t)n * p.E, n, false, sel[warp], nullptr);
        __syncwarp();
        if (lane < p.k) {
            const int e = __ldcg(p.topk_idx + (size_t)n * p.k + lane);
            if (e >= 0 && e < p.E) atomicOr(p.rbits + (size_t)(n >> 5) * p.E + e, 1u << (n & 31));
        }
        return;
    }
    if (p.x == nullptr) return;
    const int nc = (p.d + RT_CHUNK - 1) / RT_CHUNK;
    const int i = b - n_topk_ctas, n = i / nc, c = i - n * nc;
    if (n < p.N) prep_chunk_mx(p, n, c);
}

// one CTA, a thread per expert: the selected experts (ascending), each one's first
// pair, and per 32-row group the offset of the group's first pair of the expert;
// the bitmaps are moved to their copy and cleared for the next call
__global__ void __launch_bounds__(1024) route_count_kernel(const RouteParams p) {
    __shared__ int s_warp_cnt[32], s_warp_use[32];
    const int e = threadIdx.x, lane = e & 31, warp = e >> 5;
    const int G = (p.N + 31) / 32;
    int cnt = 0;
    if (e < p.E)
        for (int g = 0; g < G; g++) cnt += __popc(__ldcg(p.rbits + (size_t)g * p.E + e));
    const int use = cnt > 0 ? 1 : 0;
    // exclusive scans of the counts and of the "selected" flags over the experts
    int ic = cnt, iu = use;
    for (int o = 1; o < 32; o <<= 1) {
        const int a = __shfl_up_sync(0xffffffffu, ic, o), bu = __shfl_up_sync(0xffffffffu, iu, o);
        if (lane >= o) {
            ic += a;
            iu += bu;
        }
    }
    if (lane == 31) {
        s_warp_cnt[warp] = ic;
        s_warp_use[warp] = iu;
    }
    __syncthreads();
    if (warp == 0) {
        int wc = s_warp_cnt[lane], wu = s_warp_use[lane];
        for (int o = 1; o < 32; o <<= 1) {
            const int a = __shfl_up_sync(0xffffffffu, wc, o), bu = __shfl_up_sync(0xffffffffu, wu, o);
            if (lane >= o) {
                wc += a;
                wu += bu;
            }
        }
        s_warp_cnt[lane] = wc;
        s_warp_use[lane] = wu;
    }
    __syncthreads();
    const int before_c = (warp ? s_warp_cnt[warp - 1] : 0) + ic - cnt;
    const int before_u = (warp ? s_warp_use[warp - 1] : 0) + iu - use;
    if (e < p.E) {
        if (use) {
            p.uexp[before_u] = e;
            p.off[before_u] = before_c;
        }
        int run = before_c;
        for (int g = 0; g < G; g++) {
            const size_t at = (size_t)g * p.E + e;
            const uint32_t bits = __ldcg(p.rbits + at);
            p.rbase[at] = run;
            p.rbits2[at] = bits;
            p.rbits[at] = 0u;
            run += __popc(bits);
        }
    }
    if (e == (int)blockDim.x - 1) {
        const int U = s_warp_use[31], NK = s_warp_cnt[31];
        p.off[U] = NK;
        p.ctrl[CTRL_UNIQUE] = (uint32_t)U;
        p.ctrl[CTRL_ROWS] = (uint32_t)p.N;
        p.ctrl[CTRL_WORK] = 0;
        p.ctrl[CTRL_EXIT] = 0;
        p.ctrl[CTRL_WORK_TC] = 0;
        p.ctrl[CTRL_EXIT_TC] = 0;
    }
    for (int i = e; i < p.v_cap; i += blockDim.x) p.gu_done[i] = 0;
    for (int64_t i = e; i < p.pairs_cap; i += blockDim.x) p.hmax[i] = 0;
    if (e < RT_MAX_ROWS) p.ctrl[CTRL_XMAX + e] = 0;  // the row maxima of rows < 32 published by the prep
}

// every (row, slot) pair at its place: the expert's pairs ordered by row
__global__ void __launch_bounds__(256) route_scatter_kernel(const RouteParams p) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= p.N * p.k) return;
    const int n = i / p.k;
    const int e = __ldcg(p.topk_idx + i);
    if (e < 0 || e >= p.E) return;
    const size_t at = (size_t)(n >> 5) * p.E + e;
    const int rank = __ldcg(p.rbase + at) + __popc(__ldcg(p.rbits2 + at) & ((1u << (n & 31)) - 1u));
    p.pair[rank] = i;
}

}  // namespace moe

using namespace moe;

// ---------------------------------------------------------------------------
// router GEMM for blocks of more than 32 rows: logit[n][e] = sum_c x[n][c] Wr[e][c]
// on the tensor cores (bf16 products are exact, fp32 accumulate); the selection
// then runs on these logits as on caller logits
// ---------------------------------------------------------------------------

constexpr int RG_TM = 64;     // experts per CTA tile
constexpr int RG_TN = 64;     // rows per CTA tile
constexpr int RG_TK = 64;     // K per stage
constexpr int RG_LD = RG_TK + 8;  // padded smem row (halves): conflict-free fragment loads

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}

// D[16x8] += A[16x16] * B[16x8], bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One CTA: 64 experts x 64 rows; warp w: experts 16w..16w+15 x all 64 rows (8 MMA
// column tiles); K in stages of 64, double-buffered through cp.async.
__global__ void __launch_bounds__(128) route_gemm_kernel(int d, int E, int N, const uint16_t* __restrict__ x,
                                                         const uint16_t* __restrict__ w, float* __restrict__ logits) {
    __shared__ __align__(16) uint16_t sa[2][RG_TM * RG_LD];
    __shared__ __align__(16) uint16_t sb[2][RG_TN * RG_LD];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, i = lane & 3;
    const int e0 = blockIdx.x * RG_TM, n0 = blockIdx.y * RG_TN;
    auto load = [&](int buf, int kc) {
        // 64 rows x 128 B per operand: 512 pieces of 16 B each, 4 per thread
#pragma unroll
        for (int t = 0; t < 4; t++) {
            const int piece = tid + 128 * t, row = piece >> 3, c8 = (piece & 7) * 8;
            const int e = e0 + row, n = n0 + row;
            cp_async16(&sa[buf][row * RG_LD + c8], w + (size_t)(e < E ? e : 0) * d + kc + c8, e < E);
            cp_async16(&sb[buf][row * RG_LD + c8], x + (size_t)(n < N ? n : 0) * d + kc + c8, n < N);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    float acc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; nt++)
#pragma unroll
        for (int t = 0; t < 4; t++) acc[nt][t] = 0.f;
    const int nk = d / RG_TK;
    load(0, 0);
    for (int kc = 0; kc < nk; kc++) {
        const int buf = kc & 1;
        if (kc + 1 < nk) {
            load(buf ^ 1, (kc + 1) * RG_TK);
            asm volatile("cp.async.wait_group 1;" ::: "memory");
        } else {
            asm volatile("cp.async.wait_group 0;" ::: "memory");
        }
        __syncthreads();
        const uint16_t* A = sa[buf] + (warp * 16) * RG_LD;
        const uint16_t* Bm = sb[buf];
#pragma unroll
        for (int ks = 0; ks < RG_TK / 16; ks++) {
            const int k = ks * 16 + 2 * i;
            const uint32_t a0 = *reinterpret_cast<const uint32_t*>(A + g * RG_LD + k);
            const uint32_t a1 = *reinterpret_cast<const uint32_t*>(A + (g + 8) * RG_LD + k);
            const uint32_t a2 = *reinterpret_cast<const uint32_t*>(A + g * RG_LD + k + 8);
            const uint32_t a3 = *reinterpret_cast<const uint32_t*>(A + (g + 8) * RG_LD + k + 8);
#pragma unroll
            for (int nt = 0; nt < 8; nt++) {
                const uint32_t b0 = *reinterpret_cast<const uint32_t*>(Bm + (nt * 8 + g) * RG_LD + k);
                const uint32_t b1 = *reinterpret_cast<const uint32_t*>(Bm + (nt * 8 + g) * RG_LD + k + 8);
                mma_bf16(acc[nt], a0, a1, a2, a3, b0, b1);
            }
        }
        __syncthreads();
    }
    // C fragment: rows (experts) g and g + 8 of the warp's 16, columns (rows n) 2i, 2i + 1
#pragma unroll
    for (int nt = 0; nt < 8; nt++) {
#pragma unroll
        for (int t = 0; t < 4; t++) {
            const int e = e0 + warp * 16 + g + (t >= 2 ? 8 : 0);
            const int n = n0 + nt * 8 + 2 * i + (t & 1);
            if (e < E && n < N) logits[(size_t)n * E + e] = acc[nt][t];
        }
    }
}

extern "C" int moe_route(const moe_desc* desc, int32_t n_rows, const uint16_t* x, const uint16_t* w_router,
                         const float* logits_in, float* logits_out, int32_t* topk_idx, float* topk_w,
                         void* ws, int32_t n_rows_max, int32_t n_shared, void* stream) {
    if (!desc || !topk_idx || !topk_w || !ws) return MOE_ERR_INVALID_ARG;
    const int d = desc->d_model, f = desc->d_ff, E = desc->n_experts, k = desc->top_k;
    if (desc->group != 32 || d <= 0 || d % 256 || f <= 0 || f % 64 || E <= 0 || E > 1024 || k < 1 ||
        k > 32 || k > E)
        return MOE_ERR_UNSUPPORTED;
    if (n_rows < 1 || n_rows > n_rows_max || n_shared < 0) return MOE_ERR_UNSUPPORTED;
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
    p.rbits = reinterpret_cast<uint32_t*>(base + L.rbits);
    p.rbits2 = reinterpret_cast<uint32_t*>(base + L.rbits2);
    p.rbase = reinterpret_cast<int*>(base + L.rbase);
    p.v_cap = n_shared + (n_rows_max * k < E ? n_rows_max * k : E);
    p.pairs_cap = L.pairs;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (n_rows > RT_MAX_ROWS) {
        // prefill: the router GEMM (unless the caller gives logits), then top-k and
        // bitmaps per row (+ activation terms), counts and offsets, then every pair at
        // its place
        if (!logits_in) {
            if (d % RG_TK) return MOE_ERR_UNSUPPORTED;
            float* lg = logits_out ? logits_out : reinterpret_cast<float*>(base + L.logits);
            route_gemm_kernel<<<dim3((E + RG_TM - 1) / RG_TM, (n_rows + RG_TN - 1) / RG_TN), 128, 0, cs>>>(
                d, E, n_rows, x, w_router, lg);
            p.logits_in = lg;
        }
        p.n_ks = p.n_eg = p.n_gemv_ctas = 0;
        const int topk_ctas = (n_rows + RT_THREADS / 32 - 1) / (RT_THREADS / 32);
        const int prep = x ? n_rows * ((d + RT_CHUNK - 1) / RT_CHUNK) : 0;
        route_rows_kernel<<<topk_ctas + prep, RT_THREADS, 0, cs>>>(p, topk_ctas);
        route_count_kernel<<<1, 1024, 0, cs>>>(p);
        route_scatter_kernel<<<(n_rows * k + 255) / 256, 256, 0, cs>>>(p);
        return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
    }
    const int KS = d < RT_KS ? d : RT_KS;
    p.n_ks = d / KS;
    p.n_eg = (E + RT_EG - 1) / RT_EG;
    if (p.n_eg > 32 || p.n_ks > RT_MAX_KS) return MOE_ERR_UNSUPPORTED;
    // the partial logits and the groups' candidates must fit in the h buffer
    const size_t part_bytes = ((size_t)p.n_ks * n_rows * E * 4 + 7) & ~(size_t)7;
    if (part_bytes + (size_t)n_rows * p.n_eg * k * 8 > L.dbg_g - L.h) return MOE_ERR_UNSUPPORTED;
    p.cand = reinterpret_cast<uint64_t*>(base + L.h + part_bytes);
    p.n_gemv_ctas = logits_in ? 0 : p.n_ks * p.n_eg;
    const int prep_ctas = (logits_in && x) ? n_rows * ((d + RT_CHUNK - 1) / RT_CHUNK) : n_rows;
    int grid = p.n_gemv_ctas > prep_ctas ? p.n_gemv_ctas : prep_ctas;
    const size_t smem = (size_t)RT_MAX_ROWS * 32 * 17 * 4;  // padded x slice (also covers the grouping tables)
    static const cudaError_t attr = kernel_smem_attrs(route_kernel, (int)smem);
    if (attr != cudaSuccess) return MOE_ERR_CUDA;
    route_kernel<<<grid, RT_THREADS, smem, cs>>>(p);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
