// Block-scaled tensor-core path (tcgen05, kind::mxf8f6f4) for the routed MXFP4
// experts of a decode block.
//
// Pages: "Run Kimi 3.1 locally on one GPU": MXFP4 experts (section "One GPU,
// three storage tiers"); a block reads each expert once for all its rows
// (section "A drafter that leaves the answer unchanged").
//
// Each expert's E2M1 codes and E8M0 scales go to the tensor cores exactly as
// they are stored: TMA unpacks the 4-bit codes into the byte-per-element
// shared-memory form that kind::mxf8f6f4 reads (16U4_ALIGN16B), the scales are
// moved into tensor memory, and tcgen05.mma applies them per 32-element block.
// The activations are the other operand, each row split into three E4M3 terms
// with their own E8M0 block scales (v ~ sum of terms, about 12 bits), so a
// token is three B columns whose results are summed in a fixed order.
//
// One CTA per SM, persistent, warp-specialised:
//   warp 0      producer: claims work items in order, TMA loads (4-stage ring)
//   warp 1      one thread issues the MMAs and the commits
//   warps 2..5  move each stage's block scales from shared to tensor memory
//   warps 6..9  epilogue: read the TMEM accumulators (double-buffered), finish
//               SwiGLU and re-split h into E4M3 terms, or write the outputs.
// Work items: gate/up items (64 rows of gate + the same 64 rows of up = one
// M=128 tile, full K) and down items (128 rows, full K), ordered gate/up of
// expert v then down of expert v-4; a down item's activations are read only
// after every gate/up item of its expert has finished (bounded wait).
#include "common.cuh"

namespace moe {
namespace tc {

constexpr int NST = 4;                      // ring stages
constexpr int KC = 256;                     // K elements per stage
constexpr int NB_MAX = 48;                  // B rows: 3 terms x 16 tokens / pairs
constexpr int A_BYTES = 128 * KC;           // 128 rows x 256 codes, one byte each after unpacking
constexpr int OFF_AS = A_BYTES;             // A scales: 128 rows x 16 bytes (8 used per stage)
constexpr int OFF_B = OFF_AS + 128 * 16;    // 34816: B, two K boxes of NB_MAX rows x 128 bytes
constexpr int B_BOX = NB_MAX * 128;         // 6144
constexpr int OFF_BS = OFF_B + 2 * B_BOX;   // 47104: B scales, NB_MAX rows x 16 bytes
constexpr int STAGE = 48128;                // rounded up to 1024
constexpr int XCH_FLOATS = 128 * 16;        // gate/up exchange: 128 rows x 16 tokens
constexpr int NWARPS = 10;
constexpr int NTHREADS = NWARPS * 32;
constexpr size_t SMEM = (size_t)NST * STAGE + XCH_FLOATS * 4 + 1024 + 1024;
constexpr uint32_t TM_COLS = 256;
constexpr uint32_t TM_ACC = 0;    // accumulators: columns [0, 64) and [64, 128)
constexpr uint32_t TM_SFA = 128;  // A scales: + stage*8 + set*4 (four 32-row columns)
constexpr uint32_t TM_SFB = 160;  // B scales: same layout

enum { IT_GU = 0, IT_DN = 1 };

struct Params {
    CUtensorMap a_map[3];  // codes of gate, up, down (4-bit elements, unpacked to bytes)
    CUtensorMap s_map[3];  // E8M0 scales of gate, up, down
    CUtensorMap x_map, xs_map;  // E4M3 terms of the block's rows (row 3n+t) and their scales
    CUtensorMap h_map, hs_map;  // E4M3 terms of the pairs' SwiGLU activations (row 3P+t)
    int d, f, k, n_rows, n_shared, nbx;
    int n_gu, n_dn, lag, debug;
    const int* expert_slot;
    const uint32_t* slot_ready;
    int n_slots;
    uint32_t* ctrl;
    const int* uexp;
    const int* off;
    const int* pair;
    uint32_t* gu_done;
    uint8_t* h_mx;
    uint8_t* h_sc;
    float* y_part;
    float* dbg_g;
    float* dbg_u;
};

struct Meta {
    int item, type, u, blk, chunk, nchunks, nb, pad;
};

struct AccMeta {
    int item, type, u, blk, nb, pad[3];
};

// --- tcgen05 wrappers -------------------------------------------------------

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tm_st4(uint32_t taddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ void tm_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
          "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
}

// shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 B apart
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// instruction descriptor: E2M1 A, E4M3 B, fp32 D, K-major, M = 128, N = nb,
// E8M0 scales, scale byte `sf` of the 32-bit scale words for both operands
__device__ __forceinline__ uint32_t idesc(int nb, int sf) {
    return ((uint32_t)sf << 4) | (5u << 7) | (0u << 10) | ((uint32_t)(nb >> 3) << 17) | (1u << 23) | (8u << 24) |
           ((uint32_t)sf << 29);
}

__device__ __forceinline__ void mma_mx(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id, uint32_t sfa, uint32_t sfb,
                                       bool acc) {
    asm volatile(
        "{ .reg .pred p; setp.ne.u32 p, %6, 0;\n"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p; }" ::"r"(
            d_tmem),
        "l"(a), "l"(b), "r"(id), "r"(sfa), "r"(sfb), "r"(acc ? 1u : 0u)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 2, 128;" ::: "memory"); }

__device__ __forceinline__ int round16(int v) { return (v + 15) & ~15; }

__device__ void decode_item(const Params& p, int V, int item, int& type, int& v, int& blk) {
    int rest = item;
    for (int i = 0; i < V + p.lag; i++) {
        if (i < V) {
            if (rest < p.n_gu) {
                type = IT_GU;
                v = i;
                blk = rest;
                return;
            }
            rest -= p.n_gu;
        }
        const int vd = i - p.lag;
        if (vd >= 0 && vd < V) {
            if (rest < p.n_dn) {
                type = IT_DN;
                v = vd;
                blk = rest;
                return;
            }
            rest -= p.n_dn;
        }
    }
    type = IT_GU;
    v = 0;
    blk = 0;
}

// ---------------------------------------------------------------------------

__device__ void producer(const Params& p, int U, unsigned char* smem, uint64_t* full, uint64_t* empty, Meta* meta) {
    for (int m = 0; m < 3; m++) {
        tma_prefetch_desc(&p.a_map[m]);
        tma_prefetch_desc(&p.s_map[m]);
    }
    const int total = U * (p.n_gu + p.n_dn);
    uint32_t stage = 0, phase = 0, pending = 0, pending_par = 0;
    bool ok = true;
    while (ok) {
        const int item = (int)atomicAdd(p.ctrl + CTRL_WORK_TC, 1u);
        if (item >= total) break;
        int type, u, blk;
        decode_item(p, U, item, type, u, blk);
        const int e = __ldg(p.uexp + u);
        int z = __ldg(p.expert_slot + e);
        if (z < 0 || z >= p.n_slots) {
            set_error(p.ctrl, MOE_EBIT_BAD_SLOT);
            z = 0;
        }
        if (p.slot_ready != nullptr && ld_acquire(p.slot_ready + z) == 0u) {
            const uint64_t t0 = global_ns();
            while (ld_acquire(p.slot_ready + z) == 0u) {
                if (timed_out(p.ctrl)) break;
                if (global_ns() - t0 > WAIT_LIMIT_NS) {
                    set_error(p.ctrl, MOE_EBIT_TIMEOUT);
                    break;
                }
                __nanosleep(256);
            }
        }
        const int o0 = __ldg(p.off + u), r = __ldg(p.off + u + 1) - o0;
        if (type == IT_DN) {
            // the expert's SwiGLU activations must be complete before TMA reads them
            if (ld_acquire(p.gu_done + u) < (uint32_t)p.n_gu) {
                const uint64_t t0 = global_ns();
                while (ld_acquire(p.gu_done + u) < (uint32_t)p.n_gu) {
                    if (timed_out(p.ctrl)) break;
                    if (global_ns() - t0 > WAIT_LIMIT_NS) {
                        set_error(p.ctrl, MOE_EBIT_TIMEOUT);
                        break;
                    }
                    __nanosleep(128);
                }
            }
            asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        const bool gu = type == IT_GU;
        const int nch = (gu ? p.d : p.f) / KC;
        const int nb = gu ? p.nbx : round16(3 * r);
        const int box_rows = gu ? p.nbx : NB_MAX;
        const int brow = gu ? 0 : 3 * o0;
        const int row0 = gu ? blk * 64 : blk * 128;
        // an unpacked 4-bit code box counts its packed (global) bytes: half its shared-memory size
        const uint32_t tx = (uint32_t)(A_BYTES / 2 + 128 * 16 + 2 * box_rows * 128 + box_rows * 16);
        const CUtensorMap* bmap = gu ? &p.x_map : &p.h_map;
        const CUtensorMap* bsmap = gu ? &p.xs_map : &p.hs_map;
        for (int c = 0; c < nch; c++) {
            if (!mbar_wait(&empty[stage], phase ^ 1u)) {
                set_error(p.ctrl, MOE_EBIT_TIMEOUT);
                ok = false;
                break;
            }
            pending &= ~(1u << stage);
            Meta& mt = meta[stage];
            mt.item = item;
            mt.type = type;
            mt.u = u;
            mt.blk = blk;
            mt.chunk = c;
            mt.nchunks = nch;
            mt.nb = nb;
            mbar_arrive_expect_tx(&full[stage], tx);
            unsigned char* st = smem + (size_t)stage * STAGE;
            const int xs = (c * (KC / 32)) & ~15;  // 16-byte scale box holding this stage's 8 scale bytes
            for (int kb2 = 0; kb2 < 2; kb2++) {
                const int x = c * KC + kb2 * 128;
                if (gu) {
                    tma_load_3d(st + kb2 * 16384, &p.a_map[0], &full[stage], x, row0, z);
                    tma_load_3d(st + kb2 * 16384 + 8192, &p.a_map[1], &full[stage], x, row0, z);
                } else {
                    tma_load_3d(st + kb2 * 16384, &p.a_map[2], &full[stage], x, row0, z);
                }
                tma_load_3d(st + OFF_B + kb2 * B_BOX, bmap, &full[stage], x, brow, 0);
            }
            if (gu) {
                tma_load_3d(st + OFF_AS, &p.s_map[0], &full[stage], xs, row0, z);
                tma_load_3d(st + OFF_AS + 64 * 16, &p.s_map[1], &full[stage], xs, row0, z);
            } else {
                tma_load_3d(st + OFF_AS, &p.s_map[2], &full[stage], xs, row0, z);
            }
            tma_load_3d(st + OFF_BS, bsmap, &full[stage], xs, brow, 0);
            pending |= 1u << stage;
            pending_par = (pending_par & ~(1u << stage)) | (phase << stage);
            if (++stage == NST) {
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
    for (int s = 0; s < NST; s++)
        if (pending & (1u << s)) mbar_wait(&full[s], (pending_par >> s) & 1u);
}

// warps 2..5: each stage's E8M0 scales from shared to tensor memory.  Scale of
// row m (A: weight row, B: activation row) for the stage's K blocks 4*set..4*set+3
// is byte (kb % 4) of the 32-bit word at lane m % 32, column base + set*4 + m / 32;
// each warp writes the copy in its own lane quadrant.
__device__ void scale_mover(const Params& p, unsigned char* smem, uint32_t tbase, uint64_t* full, uint64_t* sfr,
                            const Meta* meta) {
    const int lane = threadIdx.x & 31, q = (threadIdx.x >> 5) & 3;
    uint32_t stage = 0, phase = 0;
    while (true) {
        if (!mbar_wait(&full[stage], phase)) {
            if (lane == 0) set_error(p.ctrl, MOE_EBIT_TIMEOUT);
            break;
        }
        const Meta m = meta[stage];
        if (m.item < 0) break;
        const uint32_t st = smem_u32(smem + (size_t)stage * STAGE);
        const int kb_off = (m.chunk * (KC / 32)) & 15;
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
#pragma unroll
        for (int set = 0; set < 2; set++) {
            uint32_t wa[4], wb[4];
#pragma unroll
            for (int c = 0; c < 4; c++) {
                const int row = 32 * c + lane;
                wa[c] = lds32(st + OFF_AS + row * 16 + kb_off + 4 * set);
                wb[c] = row < m.nb ? lds32(st + OFF_BS + row * 16 + kb_off + 4 * set) : 0u;
            }
            tm_st4(tbase + TM_SFA + stage * 8 + set * 4 + lane_base, wa[0], wa[1], wa[2], wa[3]);
            tm_st4(tbase + TM_SFB + stage * 8 + set * 4 + lane_base, wb[0], wb[1], wb[2], wb[3]);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sfr[stage]);
        if (++stage == NST) {
            stage = 0;
            phase ^= 1u;
        }
    }
}

// warp 1, one thread: eight MMAs (K = 32 each) per stage into the item's accumulator
__device__ void mma_issuer(const Params& p, unsigned char* smem, uint32_t tbase, uint64_t* full, uint64_t* empty,
                           uint64_t* sfr, uint64_t* acc_full, uint64_t* acc_empty, uint64_t* done, const Meta* meta,
                           AccMeta* am) {
    uint32_t stage = 0, phase = 0, it = 0;
    bool ok = true;
    while (true) {
        if (!mbar_wait(&full[stage], phase) ) {
            set_error(p.ctrl, MOE_EBIT_TIMEOUT);
            ok = false;
            break;
        }
        const Meta m = meta[stage];
        if (m.item < 0) break;
        if (!mbar_wait(&sfr[stage], phase)) {
            set_error(p.ctrl, MOE_EBIT_TIMEOUT);
            ok = false;
            break;
        }
        fence_after();
        const uint32_t b = it & 1u;
        if (m.chunk == 0) {
            if (!mbar_wait(&acc_empty[b], ((it >> 1) & 1u) ^ 1u)) {
                set_error(p.ctrl, MOE_EBIT_TIMEOUT);
                ok = false;
                break;
            }
            fence_after();
            AccMeta& a = am[b];
            a.item = m.item;
            a.type = m.type;
            a.u = m.u;
            a.blk = m.blk;
            a.nb = m.nb;
        }
        const uint32_t st = smem_u32(smem + (size_t)stage * STAGE);
#pragma unroll
        for (int ks = 0; ks < KC / 32; ks++) {
            const uint64_t ad = sdesc(st + (ks >> 2) * 16384 + (ks & 3) * 32);
            const uint64_t bd = sdesc(st + OFF_B + (ks >> 2) * B_BOX + (ks & 3) * 32);
            mma_mx(tbase + TM_ACC + b * 64, ad, bd, idesc(m.nb, ks & 3), tbase + TM_SFA + stage * 8 + (ks >> 2) * 4,
                   tbase + TM_SFB + stage * 8 + (ks >> 2) * 4, (m.chunk | ks) != 0);
        }
        mma_commit(&empty[stage]);
        if (m.chunk == m.nchunks - 1) {
            mbar_arrive(&acc_full[b]);  // publishes am[b] (release)
            mma_commit(&acc_full[b]);   // completes when the accumulator is final
            it++;
        }
        if (++stage == NST) {
            stage = 0;
            phase ^= 1u;
        }
    }
    if (ok) {  // tell the epilogue there is nothing more
        const uint32_t b = it & 1u;
        if (mbar_wait(&acc_empty[b], ((it >> 1) & 1u) ^ 1u)) {
            am[b].item = -1;
            mbar_arrive(&acc_full[b]);
            mbar_arrive(&acc_full[b]);
        } else {
            set_error(p.ctrl, MOE_EBIT_TIMEOUT);
        }
    }
    // every MMA this thread issued has completed before tensor memory is released
    mma_commit(done);
    mbar_wait(done, 0);
}

__device__ void epilogue(const Params& p, uint32_t tbase, float* xch, uint64_t* acc_full, uint64_t* acc_empty,
                         const AccMeta* am) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, q = warp & 3, ew = warp - 6;
    const int N = p.n_rows, k = p.k;
    uint32_t it = 0;
    while (true) {
        const uint32_t b = it & 1u;
        if (!mbar_wait(&acc_full[b], (it >> 1) & 1u)) {
            if (lane == 0) set_error(p.ctrl, MOE_EBIT_TIMEOUT);
            break;
        }
        fence_after();
        const AccMeta a = am[b];
        if (a.item < 0) break;
        uint32_t v[48];
        const uint32_t ta = tbase + TM_ACC + b * 64 + ((uint32_t)(32 * q) << 16);
        {
            uint32_t t16[16];
            tm_ld16(ta, t16);
#pragma unroll
            for (int i = 0; i < 16; i++) v[i] = t16[i];
            if (a.nb > 16) {
                tm_ld16(ta + 16, t16);
#pragma unroll
                for (int i = 0; i < 16; i++) v[16 + i] = t16[i];
            }
            if (a.nb > 32) {
                tm_ld16(ta + 32, t16);
#pragma unroll
                for (int i = 0; i < 16; i++) v[32 + i] = t16[i];
            }
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        }
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[b]);
        const int m = 32 * q + lane;
        const int o0 = __ldg(p.off + a.u), r = __ldg(p.off + a.u + 1) - o0;
        if (a.type == IT_GU) {
            // the 3 term columns of token n summed in order; rows 0..63 gate, 64..127 up
#pragma unroll
            for (int n = 0; n < 16; n++)
                if (n < N)
                    xch[m * 16 + n] = __uint_as_float(v[3 * n]) + __uint_as_float(v[3 * n + 1]) +
                                      __uint_as_float(v[3 * n + 2]);
            epi_sync();
            const int j0 = a.blk * 64;
            bool wrote = false;
            for (int task = ew; task < 2 * r; task += 4) {
                const int col = task >> 1, jb = task & 1;
                const int P = o0 + col;
                const int n = __ldg(p.pair + P) / k;
                const int j = 32 * jb + lane;
                const float g = xch[j * 16 + n], u = xch[(64 + j) * 16 + n];
                const float hv = g / (1.f + expf(-g)) * u;
                if (p.debug) {
                    const size_t o = (size_t)(p.n_shared * N + P) * p.f + j0 + j;
                    p.dbg_g[o] = g;
                    p.dbg_u[o] = u;
                }
                uint32_t qv[3], sb[3];
                mx3_split(hv, qv, sb);
#pragma unroll
                for (int t = 0; t < 3; t++) {
                    p.h_mx[(size_t)(3 * P + t) * p.f + j0 + j] = (uint8_t)qv[t];
                    if (lane == 0) p.h_sc[(size_t)(3 * P + t) * (p.f / 32) + (j0 >> 5) + jb] = (uint8_t)sb[t];
                }
                wrote = true;
            }
            if (wrote) __threadfence();
            epi_sync();
            if (ew == 0 && lane == 0) red_release_add(p.gu_done + a.u, 1u);
        } else {
            const int m0 = a.blk * 128;
#pragma unroll
            for (int col = 0; col < NB_MAX / 3; col++) {
                if (col < r) {
                    const float y = __uint_as_float(v[3 * col]) + __uint_as_float(v[3 * col + 1]) +
                                    __uint_as_float(v[3 * col + 2]);
                    const int pid = __ldg(p.pair + o0 + col);
                    p.y_part[(size_t)pid * p.d + m0 + m] = y;
                }
            }
        }
        it++;
    }
}

__global__ void __launch_bounds__(NTHREADS, 1) tc_expert_kernel(const __grid_constant__ Params p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    float* xch = reinterpret_cast<float*>(smem + (size_t)NST * STAGE);
    uint64_t* bars = reinterpret_cast<uint64_t*>(xch + XCH_FLOATS);
    uint64_t* full = bars;
    uint64_t* empty = full + NST;
    uint64_t* sfr = empty + NST;
    uint64_t* acc_full = sfr + NST;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* done = acc_empty + 2;
    Meta* meta = reinterpret_cast<Meta*>(done + 1);
    AccMeta* am = reinterpret_cast<AccMeta*>(meta + NST);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(am + 2);
    __shared__ int s_last;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < NST; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&sfr[s], 4);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(&acc_full[b], 2);
            mbar_init(&acc_empty[b], 4);
        }
        mbar_init(done, 1);
        mbar_fence_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                     "r"(TM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tbase = *tslot;
    const int U = (int)p.ctrl[CTRL_UNIQUE];

    if (warp == 0) {
        if (lane == 0) producer(p, U, smem, full, empty, meta);
    } else if (warp == 1) {
        if (lane == 0) mma_issuer(p, smem, tbase, full, empty, sfr, acc_full, acc_empty, done, meta, am);
    } else if (warp < 6) {
        scale_mover(p, smem, tbase, full, sfr, meta);
    } else {
        epilogue(p, tbase, xch, acc_full, acc_empty, am);
    }

    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(TM_COLS));
    // the last CTA to finish leaves the counters clean for the next call
    if (tid == 0) {
        __threadfence();
        s_last = atomicAdd(p.ctrl + CTRL_EXIT_TC, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (s_last) {
        __threadfence();
        for (int i = tid; i < U; i += NTHREADS) p.gu_done[i] = 0;
        if (tid == 0) {
            p.ctrl[CTRL_WORK_TC] = 0;
            p.ctrl[CTRL_EXIT_TC] = 0;
        }
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &qr) ==
                cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

static bool map3(CUtensorMap* m, CUtensorMapDataType type, const void* addr, uint64_t d0, uint64_t d1, uint64_t d2,
                 uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1, bool swizzle) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {s1, s2};
    const cuuint32_t box[3] = {b0, b1, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, type, 3, const_cast<void*>(addr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc

// Shapes the block-scaled path serves: both contraction lengths multiples of the
// 256-element stage, and blocks of at most 16 rows (48 activation columns).
bool tc_expert_supported(int d, int f, int n_rows) {
    return d % 256 == 0 && f % 256 == 0 && d >= 256 && f >= 256 && n_rows >= 1 && n_rows <= 16;
}

int tc_expert_launch(const moe_desc* desc, int n_rows, int mode, const moe_pool* routed, const int32_t* expert_slot,
                     const uint32_t* slot_ready, int n_shared, void* ws, int n_rows_max, float* y_part,
                     cudaStream_t stream) {
    using namespace tc;
    const int d = desc->d_model, f = desc->d_ff, E = desc->n_experts, k = desc->top_k;
    const WsLayout L = ws_layout(d, f, E, k, n_rows_max, n_shared);
    char* base = static_cast<char*>(ws);
    static Params p;
    memset(&p, 0, sizeof(p));
    const char* pool = static_cast<const char*>(routed->base);
    const int64_t per = (int64_t)f * d / 2 + (int64_t)f * (d / 32);
    const char* planes_c[3] = {pool, pool + per, pool + 2 * per};
    const char* planes_s[3] = {pool + (int64_t)f * d / 2, pool + per + (int64_t)f * d / 2,
                               pool + 2 * per + (int64_t)d * f / 2};
    const int rows[3] = {f, f, d}, kk[3] = {d, d, f}, brows[3] = {64, 64, 128};
    for (int m = 0; m < 3; m++) {
        if (!map3(&p.a_map[m], CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, planes_c[m], kk[m], rows[m], routed->n_slots,
                  kk[m] / 2, routed->slot_bytes, 128, brows[m], true))
            return MOE_ERR_UNSUPPORTED;
        if (!map3(&p.s_map[m], CU_TENSOR_MAP_DATA_TYPE_UINT8, planes_s[m], kk[m] / 32, rows[m], routed->n_slots,
                  kk[m] / 32, routed->slot_bytes, 16, brows[m], false))
            return MOE_ERR_UNSUPPORTED;
    }
    const int nbx = ((3 * n_rows + 15) / 16) * 16;
    const uint64_t rx = L.mx_rows_x, rh = L.mx_rows_h;
    if (!map3(&p.x_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, base + L.x_mx, d, rx, 1, d, rx * d, 128, nbx, true) ||
        !map3(&p.xs_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, base + L.x_sc, d / 32, rx, 1, d / 32, rx * (d / 32), 16, nbx,
              false) ||
        !map3(&p.h_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, base + L.h_mx, f, rh, 1, f, rh * f, 128, NB_MAX, true) ||
        !map3(&p.hs_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, base + L.h_sc, f / 32, rh, 1, f / 32, rh * (f / 32), 16, NB_MAX,
              false))
        return MOE_ERR_UNSUPPORTED;
    p.d = d;
    p.f = f;
    p.k = k;
    p.n_rows = n_rows;
    p.n_shared = n_shared;
    p.nbx = nbx;
    p.n_gu = f / 64;
    p.n_dn = d / 128;
    p.lag = 4;
    p.debug = (mode & MOE_MODE_DEBUG_GU) ? 1 : 0;

    p.expert_slot = expert_slot;
    p.slot_ready = slot_ready;
    p.n_slots = routed->n_slots;
    p.ctrl = reinterpret_cast<uint32_t*>(base + L.ctrl);
    p.uexp = reinterpret_cast<const int*>(base + L.uexp);
    p.off = reinterpret_cast<const int*>(base + L.off);
    p.pair = reinterpret_cast<const int*>(base + L.pair);
    p.gu_done = reinterpret_cast<uint32_t*>(base + L.gu_done_tc);
    p.h_mx = reinterpret_cast<uint8_t*>(base + L.h_mx);
    p.h_sc = reinterpret_cast<uint8_t*>(base + L.h_sc);
    p.y_part = y_part;
    p.dbg_g = reinterpret_cast<float*>(base + L.dbg_g);
    p.dbg_u = reinterpret_cast<float*>(base + L.dbg_u);
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(tc_expert_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM) !=
            cudaSuccess)
            return MOE_ERR_CUDA;
        attr = true;
    }
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return MOE_ERR_CUDA;
    tc_expert_kernel<<<sms, NTHREADS, SMEM, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
