// Internal helpers of the GB300 MoE library: inline PTX wrappers (mbarrier, TMA,
// tensor-core MMA, E2M1 conversion), bounded waits, and the workspace layout.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// ---------------------------------------------------------------------------
// workspace layout (shared by host and device code)
// ---------------------------------------------------------------------------

// control words at the start of the workspace
enum Ctrl : int {
    CTRL_ERROR = 0,      // device error word (MOE_EBIT_*)
    CTRL_WORK = 1,       // next work item of the expert kernel
    CTRL_EXIT = 2,       // CTAs of the expert kernel that finished
    CTRL_TICKET = 3,     // CTAs of the route kernel that finished
    CTRL_UNIQUE = 4,     // U: experts selected by the block
    CTRL_ROWS = 5,       // rows of the routed block
    CTRL_WORK_TC = 6,    // next work item of the block-scaled tensor-core expert kernel
    CTRL_EXIT_TC = 7,    // its finished CTAs
    CTRL_WORK_SH = 8,    // next work item of the shared-expert call (runs beside routing)
    CTRL_EXIT_SH = 9,    // its finished CTAs
    CTRL_PREP_SH = 10,   // rows of the block claimed for the shared experts' f16 copy
    CTRL_PREPD_SH = 11,  // rows of that copy written
    CTRL_RT_DONE = 12,   // routing finishers done with their rows' f16 copies
    CTRL_EPOCH_TC = 13,  // launches of the block-scaled expert kernel on this workspace (tags its partial sums)
    CTRL_XMAX = 64,      // [64, 96): per-row max |x| bits published by the router GEMV CTAs
    CTRL_TL = 96,        // [96, 128): kernel timeline, 4 kernels x (~first start, last end) as u64 pairs
    CTRL_WORDS = 128
};

// position p of the routed experts' work order -> index into uexp/off (MOE_MODE_ORDERED),
// clamped into [0, U) so that a malformed order stays in bounds
__device__ __forceinline__ int ordered_index(const int* order, int u, int U) {
    if (order == nullptr) return u;
    const int v = __ldcg(order + u);
    return v < 0 ? 0 : (v >= U ? U - 1 : v);
}

// kernels of the timeline (CTRL_TL)
enum TlKernel : int { TL_ROUTE = 0, TL_SHARED = 1, TL_ROUTED = 2 };

// K splits of a gate/up tile in the block-scaled tensor-core expert kernel
constexpr int TC_GU_SPLIT = 2;
// E2M1 terms an activation value is split into for that kernel (each term with
// its own E8M0 scale per 32 elements): about 16 significant bits survive
constexpr int MX_TERMS = 5;
// K slices of the shared experts' gate/up projection
constexpr int SH_K_SPLIT = 4;

struct WsLayout {
    size_t ctrl, uexp, uorder, off, pair, x16, xexp, gu_done, hmax, h, dbg_g, dbg_u, shared_y, logits,
        x_mx, x_sc, h_mx, h_sc, gu_done_tc, gu_part, gu_state, x16s, xexps, gu_done_sh, hmax_sh, h_sh, h_sh_hl, sh_part,
        sh_cnt, rbits, rbits2, rbase, total;
    int64_t mx_rows_x, mx_rows_h;  // rows of the MX activation buffers (with padding)
    int64_t pairs;   // capacity of the pair-indexed buffers: n_shared*N + N*k
};

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

inline WsLayout ws_layout(int d, int f, int E, int k, int n_rows_max, int n_shared) {
    WsLayout L;
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 256); return at; };
    const int64_t N = n_rows_max;
    L.pairs = (int64_t)n_shared * N + N * k;
    const int64_t V = n_shared + (N * k < E ? N * k : E);
    L.ctrl = take(CTRL_WORDS * 4);
    L.uexp = take((size_t)E * 4);
    L.uorder = take((size_t)E * 4);
    L.off = take((size_t)(E + 1) * 4);
    L.pair = take((size_t)N * k * 4);
    L.x16 = take((size_t)N * d * 2);
    L.xexp = take((size_t)N * 4);
    L.gu_done = take((size_t)V * 4);
    L.hmax = take((size_t)L.pairs * 4);
    L.h = take((size_t)L.pairs * f * 4);
    L.dbg_g = take((size_t)L.pairs * f * 4);
    L.dbg_u = take((size_t)L.pairs * f * 4);
    L.shared_y = take((size_t)n_shared * N * d * 4);
    L.logits = take((size_t)N * E * 4);
    // MX activations for the block-scaled expert kernel: MX_TERMS rows of packed
    // E2M1 codes (two per byte, even element in the low nibble) per row of x and
    // per routed pair of h, plus 80 rows of padding
    L.mx_rows_x = (int64_t)MX_TERMS * N + 80;
    L.mx_rows_h = (int64_t)MX_TERMS * N * k + 80;
    L.x_mx = take((size_t)L.mx_rows_x * (d / 2));
    L.x_sc = take((size_t)L.mx_rows_x * (d / 32));
    L.h_mx = take((size_t)L.mx_rows_h * (f / 2));
    L.h_sc = take((size_t)L.mx_rows_h * (f / 32));
    // the block-scaled kernel works on chunks of at most 16 (prefill) or 6 (blocks of up
    // to 16 rows) pairs of one expert: fewer than E + N*k of them; one finished-tile
    // counter per chunk
    const int64_t chunks = E + N * k;
    L.gu_done_tc = take((size_t)chunks * 4);
    // split-K gate/up partial sums: [f/64 tiles][TC_GU_SPLIT][routed pairs][64 gate + 64
    // up] 8-byte words, each a float and the tag of the launch that wrote it, and per
    // (chunk, tile) the bits of the splits that published their sums
    L.gu_part = take((size_t)(f / 64) * TC_GU_SPLIT * (N * k) * 128 * 8);
    L.gu_state = take((size_t)chunks * (f / 64) * 4);
    // the shared-expert call's own activation copy and counters: it runs beside
    // the routing kernel, which resets the layer's counters
    L.x16s = take((size_t)N * d * 2);
    L.xexps = take((size_t)N * 4);
    L.gu_done_sh = take(64 * 4);
    L.hmax_sh = take((size_t)(n_shared > 0 ? n_shared : 1) * N * 4);
    L.h_sh = take((size_t)(n_shared > 0 ? n_shared : 1) * N * f * 4);
    // blocks of more than 16 rows: h * 2^-p of every shared pair as f16 hi and lo parts
    // ([s][N][f] each), split once for all the down projection's row tiles
    L.h_sh_hl = take((size_t)(n_shared > 0 ? n_shared : 1) * N * f * 4);
    // the shared experts' gate/up partial sums [s][f/16 tiles][32-row chunks][K slices][2][16][32]
    // and per (s, tile, chunk) the slices finished
    // (chunks of 32 block rows: 2 x 16 x 32 sums per unit and slice)
    const int64_t sh_units = (int64_t)(n_shared > 0 ? n_shared : 1) * (f / 16) * ((N + 31) / 32);
    L.sh_part = take((size_t)sh_units * SH_K_SPLIT * 1024 * 4);
    L.sh_cnt = take((size_t)sh_units * 4);
    // grouping of blocks of more than 32 rows: per (32-row group, expert) the bitmap
    // of rows that selected it (zeroed again after use), its copy, and the offset of
    // the group's first pair of the expert
    const int64_t groups = (N + 31) / 32;
    L.rbits = take((size_t)groups * E * 4);
    L.rbits2 = take((size_t)groups * E * 4);
    L.rbase = take((size_t)groups * E * 4);
    L.total = o;
    return L;
}

// Dynamic shared memory above the default limit for a kernel.
template <class K>
inline cudaError_t kernel_smem_attrs(K* kernel, int dyn) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
}

// Launch that may be scheduled before the previous kernel on the stream has
// completed (programmatic dependent launch).  Every kernel launched this way runs
// griddep_wait() before it touches memory the previous kernel writes or reads, so
// the stream order of memory effects is that of a plain launch; what overlaps is
// the launch itself and the kernel's set-up (barriers, tensor memory).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_chained(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                  Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------

// Upper bound of every spin in device code: 2 s of %globaltimer.
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Programmatic dependent launch: wait until the kernels this grid depends on have
// completed and their memory is visible (returns at once for a plain launch) ...
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ... and let the next kernel on the stream be scheduled (it still waits for this
// grid's completion before it reads anything).
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// Kernel timeline: every CTA of kernel `k` records its start and end time
// (%globaltimer, ns); the workspace keeps the bitwise complement of the earliest
// start and the latest end since the words were last zeroed (zero = none yet).
__device__ __forceinline__ void tl_begin(uint32_t* ctrl, int k) {
    atomicMax(reinterpret_cast<unsigned long long*>(ctrl + CTRL_TL) + 2 * k, (unsigned long long)~global_ns());
}
__device__ __forceinline__ void tl_end(uint32_t* ctrl, int k) {
    atomicMax(reinterpret_cast<unsigned long long*>(ctrl + CTRL_TL) + 2 * k + 1, (unsigned long long)global_ns());
}

__device__ __forceinline__ void set_error(uint32_t* ctrl, uint32_t bits) {
    atomicOr(ctrl + CTRL_ERROR, bits);
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ bool timed_out(const uint32_t* ctrl) {
    return (ld_acquire(ctrl + CTRL_ERROR) & MOE_EBIT_TIMEOUT) != 0u;
}

__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// --- mbarrier ---------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking: has the phase with the given parity of `bar` completed?
__device__ __forceinline__ bool mbar_peek(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits until the phase with the given parity of `bar` has completed; gives up
// after WAIT_LIMIT_NS and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    if (mbar_test(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (true) {
        if (mbar_test(bar, parity)) return true;
        if (global_ns() - t0 > WAIT_LIMIT_NS) return false;
    }
}

// --- TMA ------------------------------------------------------------------

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int x,
                                            int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y, int z,
                                            int w) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z), "r"(w)
        : "memory");
}

__device__ __forceinline__ void tma_load_5d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1, int c2,
                                            int c3, int c4) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
        : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// --- named barrier among the consumer warps -------------------------------

template <int NTHREADS>
__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(NTHREADS) : "memory");
}

// --- numeric conversions ----------------------------------------------------

// Two E2M1 codes (one byte, even element in the low nibble) -> f16x2 (low half = even).
// The conversion is exact: every E2M1 value is an f16 value.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t& d0, uint32_t& d1, uint32_t& d2,
                                                uint32_t& d3) {
    asm("{ .reg .b8 b0, b1, b2, b3;\n"
        "  mov.b32 {b0, b1, b2, b3}, %4;\n"
        "  cvt.rn.f16x2.e2m1x2 %0, b0;\n"
        "  cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        "  cvt.rn.f16x2.e2m1x2 %2, b2;\n"
        "  cvt.rn.f16x2.e2m1x2 %3, b3; }"
        : "=r"(d0), "=r"(d1), "=r"(d2), "=r"(d3)
        : "r"(w));
}

// Four int8 values -> two f16x2 (exact): place (v + 128) in the mantissa of
// 1024.0 and subtract 1152.
__device__ __forceinline__ void s8x4_to_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t t = w ^ 0x80808080u;
    uint32_t a, b;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(a) : "r"(t), "r"(0x64646464u), "r"(0x4140u));
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(b) : "r"(t), "r"(0x64646464u), "r"(0x4342u));
    asm("sub.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(0x64806480u));
    asm("sub.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(0x64806480u));
}

// E8M0 scale byte -> 2^(s-127) as fp32 (s = 0 is the subnormal 2^-127, 255 is NaN).
__device__ __forceinline__ float e8m0_to_f32(uint32_t s) {
    uint32_t b = s << 23;
    b = (s == 0u) ? 0x00400000u : b;
    b = (s == 255u) ? 0x7fc00000u : b;
    return __uint_as_float(b);
}

// 2^e as fp32 for e in [-126, 127].
__device__ __forceinline__ float exp2i(int e) { return __uint_as_float((uint32_t)(127 + e) << 23); }

// Scale exponent p for a row whose largest magnitude has bit pattern `maxbits`:
// max * 2^-p lands in [2^14, 2^15), inside the f16 range with room for rounding.
__device__ __forceinline__ int f16_scale_exponent(uint32_t maxbits) {
    if (maxbits == 0u) return 0;
    int e = (int)((maxbits >> 23) & 0xFFu) - 127;
    int p = e - 14;
    p = p < -100 ? -100 : p;
    p = p > 100 ? 100 : p;
    return p;
}

// One E4M3 code of v (round to nearest even, saturating) and its exact value.
__device__ __forceinline__ uint32_t e4m3_code(float v, float& back) {
    uint16_t pair;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(pair) : "f"(v));
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pair));
    back = __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
    return pair & 0xFFu;
}

// Splits the 32 values of a block (one per lane) into three E4M3 terms with their
// own power-of-two block scales, v ~ sum_t q_t * 2^(s_t - 127): each term codes the
// residual of the previous ones, so about 12 significant bits survive.  Writes the
// lane's three codes and, in every lane, the three E8M0 scale bytes.
__device__ __forceinline__ void mx3_split(float v, uint32_t (&q)[3], uint32_t (&sbyte)[3]) {
    float r = v;
#pragma unroll
    for (int t = 0; t < 3; t++) {
        const uint32_t m = __reduce_max_sync(0xffffffffu, __float_as_uint(r) & 0x7FFFFFFFu);
        int e = (int)(m >> 23) - 127 - 7;  // |r| / 2^e < 256 <= 448
        e = m == 0u ? 0 : e;
        e = e < -126 ? -126 : (e > 127 ? 127 : e);
        float back;
        q[t] = e4m3_code(r * exp2i(-e), back);
        r -= back * exp2i(e);
        sbyte[t] = (uint32_t)(e + 127);
    }
}

// E2M1 code of v (round to nearest even, saturating at +-6) and its exact value.
__device__ __forceinline__ uint32_t e2m1_code(float v, float& back) {
    uint32_t bytes, h2;
    asm("{ .reg .b8 t;\n"
        "  cvt.rn.satfinite.e2m1x2.f32 t, %2, %2;\n"
        "  cvt.rn.f16x2.e2m1x2 %1, t;\n"
        "  mov.b32 %0, {t, t, t, t}; }"
        : "=r"(bytes), "=r"(h2)
        : "f"(v));
    back = __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
    return bytes & 0xFu;
}

// Splits the 32 values of a block (one per lane) into MX_TERMS E2M1 terms with
// their own power-of-two block scales, v ~ sum_t q_t * 2^(s_t - 127): each term
// codes the residual of the previous ones (the block's largest residual lands in
// (3, 6]).  Writes the lane's codes and, in every lane, the E8M0 scale bytes.
__device__ __forceinline__ void mx_split(float v, uint32_t (&q)[MX_TERMS], uint32_t (&sbyte)[MX_TERMS]) {
    float r = v;
#pragma unroll
    for (int t = 0; t < MX_TERMS; t++) {
        const uint32_t m = __reduce_max_sync(0xffffffffu, __float_as_uint(r) & 0x7FFFFFFFu);
        // m = 1.f * 2^E: scale 2^(E-2) when f <= 1.5 (m / scale in [4, 6]), else 2^(E-1)
        int e = (int)(m >> 23) - 127 - 1 - ((m & 0x7FFFFFu) <= 0x400000u ? 1 : 0);
        e = m == 0u ? 0 : e;
        e = e < -126 ? -126 : (e > 127 ? 127 : e);
        float back;
        q[t] = e2m1_code(r * exp2i(-e), back);
        r -= back * exp2i(e);
        sbyte[t] = (uint32_t)(e + 127);
    }
}

// Stores the 32 four-bit codes of a warp (lane i: element i) as 16 packed bytes
// (even element in the low nibble) at dst, 4-byte aligned.
__device__ __forceinline__ void store_e2m1_block(uint8_t* dst, uint32_t code) {
    const int lane = threadIdx.x & 31;
    const uint32_t b = code | (__shfl_down_sync(0xffffffffu, code, 1) << 4);  // even lanes: one byte
    const uint32_t b1 = __shfl_down_sync(0xffffffffu, b, 2);
    const uint32_t b2 = __shfl_down_sync(0xffffffffu, b, 4);
    const uint32_t b3 = __shfl_down_sync(0xffffffffu, b, 6);
    if ((lane & 7) == 0)
        *reinterpret_cast<uint32_t*>(dst + (lane >> 1)) = (b & 0xFFu) | ((b1 & 0xFFu) << 8) | ((b2 & 0xFFu) << 16) |
                                                           ((b3 & 0xFFu) << 24);
}

// D[16x8] += A[16x16] * B[16x8], f16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t lds8(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t lds16(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

// the shared experts (shared.cu): from the routing kernel's f16 rows (prep = false)
// or from x through the preparation kernel (prep = true)
int shared_launch(const moe_desc* desc, int n_rows, int n_rows_max, const uint16_t* x, const moe_pool* shared,
                  int n_shared, void* ws, bool prep, bool wait_first, cudaStream_t s);

// the block-scaled tensor-core path for routed MXFP4 experts (experts_tc.cu)
bool tc_expert_supported(int d, int f, int n_rows);
int tc_expert_launch(const moe_desc* desc, int n_rows, int mode, const moe_pool* routed, const int32_t* expert_slot,
                     const uint32_t* slot_ready, int n_shared, void* ws, int n_rows_max, float* y_part,
                     cudaStream_t stream);

}  // namespace moe
