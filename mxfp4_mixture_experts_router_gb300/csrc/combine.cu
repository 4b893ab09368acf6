// Weighted combine of a block's expert outputs into the residual, and the
// host-side workspace utilities.
//
// out[n][c] = bf16_rne(residual[n][c] + (sum_j w[n][j] * y[n][j][c] + sum_s shared_s[n][c]))
// with the sum taken in slot order, then shared-expert order: a fixed order per
// element, so the result of a row does not depend on the rest of its block.
// Pages: "Run Kimi 3.1 locally on one GPU" (16 routed experts per token) and
// "Run Kimi K3 and K3.1 Pro Locally" (plus 2 shared experts).
#include "common.cuh"

namespace moe {

constexpr int CB_THREADS = 64;

// One thread per 4 consecutive columns of a row; every slot's load is issued
// before the fixed-order sum, so the loads overlap.
template <int KMAX>
__global__ void __launch_bounds__(CB_THREADS) combine_kernel(int d, int k, int n_shared, int N,
                                                             const uint16_t* __restrict__ residual,
                                                             const float* __restrict__ y_part,
                                                             const float* __restrict__ topk_w,
                                                             const float* __restrict__ shared_y,
                                                             uint16_t* __restrict__ out) {
    griddep_wait();  // launched while the expert kernels finish
    const int n = blockIdx.y;
    const int c = (blockIdx.x * CB_THREADS + threadIdx.x) * 4;
    if (c >= d) return;
    const float* yr = y_part + (size_t)n * k * d + c;
    float4 y[KMAX];
    float w[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; j++) {
        if (j < k) {
            w[j] = __ldg(topk_w + (size_t)n * k + j);
            y[j] = __ldg(reinterpret_cast<const float4*>(yr + (size_t)j * d));
        }
    }
    const uint2 rb = __ldg(reinterpret_cast<const uint2*>(residual + (size_t)n * d + c));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < KMAX; j++) {
        if (j < k) {
            acc.x = fmaf(w[j], y[j].x, acc.x);
            acc.y = fmaf(w[j], y[j].y, acc.y);
            acc.z = fmaf(w[j], y[j].z, acc.z);
            acc.w = fmaf(w[j], y[j].w, acc.w);
        }
    }
    for (int s = 0; s < n_shared; s++) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(shared_y + ((size_t)s * N + n) * d + c));
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
    }
    const float r0 = __uint_as_float(rb.x << 16), r1 = __uint_as_float(rb.x & 0xFFFF0000u);
    const float r2 = __uint_as_float(rb.y << 16), r3 = __uint_as_float(rb.y & 0xFFFF0000u);
    const __nv_bfloat16 o0 = __float2bfloat16_rn(r0 + acc.x), o1 = __float2bfloat16_rn(r1 + acc.y);
    const __nv_bfloat16 o2 = __float2bfloat16_rn(r2 + acc.z), o3 = __float2bfloat16_rn(r3 + acc.w);
    uint2 ob;
    ob.x = (uint32_t)__bfloat16_as_ushort(o0) | ((uint32_t)__bfloat16_as_ushort(o1) << 16);
    ob.y = (uint32_t)__bfloat16_as_ushort(o2) | ((uint32_t)__bfloat16_as_ushort(o3) << 16);
    *reinterpret_cast<uint2*>(out + (size_t)n * d + c) = ob;
}

}  // namespace moe

using namespace moe;

extern "C" int moe_combine(const moe_desc* desc, int32_t n_rows, const uint16_t* residual, const float* y_part,
                           const float* topk_w, const float* shared_y, int32_t n_shared, uint16_t* out,
                           void* stream) {
    if (!desc || !residual || !y_part || !topk_w || !out) return MOE_ERR_INVALID_ARG;
    if (n_shared < 0 || (n_shared > 0 && !shared_y)) return MOE_ERR_INVALID_ARG;
    const int d = desc->d_model, k = desc->top_k;
    if (d <= 0 || d % 256 || k < 1 || k > 32 || n_rows < 1) return MOE_ERR_UNSUPPORTED;
    if (((uintptr_t)residual & 7) || ((uintptr_t)out & 7) || ((uintptr_t)y_part & 15) ||
        (shared_y && ((uintptr_t)shared_y & 15)))
        return MOE_ERR_INVALID_ARG;
    dim3 grid((d / 4 + CB_THREADS - 1) / CB_THREADS, n_rows);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const cudaError_t e =
        k <= 16 ? launch_chained(combine_kernel<16>, grid, dim3(CB_THREADS), 0, s, d, k, n_shared, (int)n_rows, residual,
                                 y_part, topk_w, shared_y, out)
                : launch_chained(combine_kernel<32>, grid, dim3(CB_THREADS), 0, s, d, k, n_shared, (int)n_rows, residual,
                                 y_part, topk_w, shared_y, out);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" size_t moe_workspace_size(const moe_desc* desc, int32_t n_rows_max, int32_t n_shared) {
    if (!desc || n_rows_max < 1 || n_shared < 0) return 0;
    return ws_layout(desc->d_model, desc->d_ff, desc->n_experts, desc->top_k, n_rows_max, n_shared).total;
}

extern "C" int moe_workspace_offsets(const moe_desc* desc, int32_t n_rows_max, int32_t n_shared,
                                     moe_ws_offsets* o) {
    if (!desc || !o || n_rows_max < 1 || n_shared < 0) return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(desc->d_model, desc->d_ff, desc->n_experts, desc->top_k, n_rows_max, n_shared);
    o->error_word = (int64_t)L.ctrl + 4 * CTRL_ERROR;
    o->n_unique = (int64_t)L.ctrl + 4 * CTRL_UNIQUE;
    o->uexp = (int64_t)L.uexp;
    o->uorder = (int64_t)L.uorder;
    o->off = (int64_t)L.off;
    o->pair = (int64_t)L.pair;
    o->dbg_g = (int64_t)L.dbg_g;
    o->dbg_u = (int64_t)L.dbg_u;
    o->h = (int64_t)L.h;
    o->shared_y = (int64_t)L.shared_y;
    o->timeline = (int64_t)L.ctrl + 4 * CTRL_TL;
    return MOE_OK;
}

extern "C" int moe_get_error(void* ws, void* stream, uint32_t* bits) {
    if (!ws || !bits) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t* word = reinterpret_cast<uint32_t*>(ws) + CTRL_ERROR;
    if (cudaMemcpyAsync(bits, word, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemsetAsync(word, 0, 4, s) != cudaSuccess) return MOE_ERR_CUDA;
    return cudaStreamSynchronize(s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
