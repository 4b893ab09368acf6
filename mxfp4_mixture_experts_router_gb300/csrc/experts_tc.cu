// Block-scaled tensor-core path (tcgen05, kind::mxf4) for the routed MXFP4
// experts of a block (decode blocks and prefill).
//
// Pages: "Run Kimi 3.1 locally on one GPU": MXFP4 experts (section "One GPU,
// three storage tiers"); a block reads each expert once for all its rows
// (section "A drafter that leaves the answer unchanged").
//
// Each expert's E2M1 codes and E8M0 scales go to the tensor cores exactly as
// they are stored: TMA copies the packed 4-bit codes into shared memory (two
// per byte, the layout kind::mxf4 reads), the scales are moved into tensor
// memory, and tcgen05.mma applies them per 32-element block (scale_vec::2X).
// The activations are the other operand, each row split into MX_TERMS E2M1
// terms with their own E8M0 block scales (v ~ sum of terms), so a token is
// MX_TERMS B columns whose results are summed in a fixed order.
//
// One CTA per SM, persistent, warp-specialised:
//   warp 0      producer: claims work items in order and TMA-loads them into a
//               ring of shared-memory stages
//   warp 1      one thread issues the MMAs and the commits
//   warps 2..    load each stage's activation rows (4 warps for decode blocks, 8
//               for prefill); warps 2..5 also load its scales and move the block
//               scales to tensor memory
//   last 4 warps epilogue: read the TMEM accumulators (double-buffered), reduce
//               the K splits of a gate/up tile, finish SwiGLU and re-split h into
//               E2M1 terms, or write the outputs.
// Work items: gate/up items (64 rows of gate + the same 64 rows of up = one
// M=128 tile, over one of TC_GU_SPLIT K ranges) and down items (128 rows, full
// K): the gate/up items of every chunk first, then the down items in chunk
// order, so a chunk's down items are claimed long after its gate/up tiles and
// none waits at the end of the launch.  A down item's activations are read
// only after every gate/up tile of its chunk is finished (bounded wait).
//
// TMA costs a roughly fixed time per box, so it carries only the weights: a
// stage is one 16 KB box of code rows (128 rows x 256 K; gate and up rows arrive
// through a 5-D tensor map) and the scales of a whole item arrive in one box into
// a per-item buffer.  Packed codes take half the shared memory (and half the
// tensor core's shared-memory reads) of the byte-per-element form, so the ring
// holds twice the stages.  The small activation operand (rows of the block or of the expert's
// pairs, from L2) and its scales are loaded by the scale-mover warps one stage
// ahead into registers (two stages ahead into L1) and written in the swizzled
// layout the MMA reads.  Every expert's slot and pair range sit in shared memory
// (read by all threads at the start), and the next item's claim is issued and
// decoded while the current item streams.
#include "common.cuh"

namespace moe {
namespace tc {

constexpr int KC = 512;                     // K elements per stage
constexpr int KCH = KC / 256;               // 128-byte pieces (256 packed K) of a row per stage
constexpr int A_BYTES = 128 * KC / 2;       // 128 rows x KC packed E2M1 codes: KCH regions of 128 x 128 B
constexpr int SF_COLS = KC / 32;            // tensor-memory scale columns per stage (4 per 128 K)
constexpr int T = MX_TERMS;                 // B columns (activation terms) per token
constexpr int SC_MAX = 112;                 // scale bytes per row of one item (its K range / 32)
constexpr int SA_BYTES = 128 * SC_MAX;      // A scales of an item
constexpr int XCH_FLOATS = 128 * 16;        // gate/up exchange: 128 rows x 16 tokens (xor-swizzled)
constexpr int CHUNK = 16;                   // most pairs of one expert per work item (80 MMA columns)
constexpr int S = TC_GU_SPLIT;
static_assert(S == 2, "the gate/up hand-over pairs exactly two splits");

// Two configurations, both with a 3-stage ring: blocks of up to 16 rows (32
// activation rows, chunks of up to 6 pairs) and prefill (80 activation rows, chunks
// of up to 16 pairs).  The 80-row configuration costs about 20 % more per byte on
// small blocks (1 row: 121 against 101 us for the layer), so decode blocks take the
// 32-row one and split an expert with more than 6 pairs into several chunks.  Three
// 40 KB stages per SM stream the weights as fast as four did, and the fewer bytes
// in flight shorten every other memory round trip of the launch (the hand-overs
// from gate/up to down items, the claims).
template <int NBM>
struct Cfg {
    static constexpr int NST = 3;                      // ring stages
    static constexpr int B_BYTES = KCH * NBM * 128;    // B of a stage: KCH regions of NBM rows x 128 B
    static constexpr int STAGE = A_BYTES + B_BYTES;    // a multiple of 1024
    static constexpr int SCB = SA_BYTES;               // one per-item A-scale buffer (two, by item parity)
    // tensor memory: two accumulator sets (double-buffered across items), each of
    // NACC accumulators that take the stage's MMAs in turn (independent MMAs
    // overlap in the tensor pipe; the epilogue sums them in order; the same NACC
    // in both configurations keeps a row's arithmetic independent of the block),
    // then the A and B scale columns of every stage
    static constexpr int ACC_COLS = NBM;
    static constexpr int NACC = 2;
    static constexpr uint32_t ACC_SET = NACC * ACC_COLS;
    static constexpr uint32_t TM_SFA = 2 * ACC_SET;    // A scales: + stage*SF_COLS + set*4 (four 32-row columns)
    static constexpr uint32_t TM_SFB = TM_SFA + NST * SF_COLS;
    static constexpr uint32_t TM_COLS = TM_SFB + NST * SF_COLS <= 256 ? 256 : 512;
    // per expert: (slot, first pair | pairs << 16) and the prefix of its chunk counts
    static constexpr int CH = NBM / T;                 // pairs per chunk: 6 (32 columns) or 16 (80)
    static constexpr int MAX_U = NBM == 32 ? 256 : 1024;
    // blocks of up to 5 rows: the block row of every (row, slot) pair (5 x k <= 160);
    // then the block rows of the pairs of the chunks in the two scale buffers' items
    static constexpr int TOKS = NBM == 32 ? 256 : 0;
    static constexpr int META_BYTES = MAX_U * 8 + (MAX_U + 1) * 4 + TOKS * 2 + 2 * CHUNK * 2 + 12;
    // each scale-mover warp's staging of the activation scale bytes, per stage
    static constexpr int SBS_BYTES = 4 * NST * NBM * 16;
    // activation-copy warps (2 .. 1 + NMOV; the first four also move the scales), then
    // four epilogue warps.  A prefill stage carries 80 activation rows, whose copies
    // take eight warps to issue; the 32-row configuration keeps four.
    static constexpr int NMOV = NBM == 32 ? 4 : 8;
    static constexpr int MOV_T = 32 * NMOV;     // copy threads
    static constexpr int EPI_W0 = 2 + NMOV;     // first epilogue warp
    static constexpr int NTHREADS = (EPI_W0 + 4) * 32;
    static constexpr size_t SMEM =
        (size_t)NST * STAGE + 2 * SCB + SBS_BYTES + XCH_FLOATS * 4 + META_BYTES + 1024 + 1024;
    static_assert(STAGE % 1024 == 0 && SCB % 128 == 0, "TMA destinations stay aligned");
    static_assert(SMEM <= 232448, "shared memory per CTA");
    static_assert(TM_SFB + NST * SF_COLS <= TM_COLS && NBM <= ACC_COLS && NBM <= 128, "tensor memory columns");
    static_assert(NBM % 16 == 0 && CHUNK * T <= 80 && CH <= CHUNK && ((CH * T + 15) & ~15) <= NBM, "MMA N");
};

enum { IT_GU = 0, IT_DN = 1 };

struct Params {
    CUtensorMap a_gu;       // gate and up codes {128 B = 256 K, f rows, 2 matrices, d/256, slot}, packed
    CUtensorMap a_dn;       // down codes {128 B, d rows, f/256, slot}
    CUtensorMap s_gu;       // gate and up E8M0 scales {d/32, f rows, 2, slot}
    CUtensorMap s_dn;       // down scales {f/32, d rows, slot}
    int d, f, k, n_rows, n_shared, nk;
    int n_gu, n_dn, lag, debug;
    int after_shared;  // launched right behind the shared experts that ran beside the routing
    const int* expert_slot;
    const uint32_t* slot_ready;
    int n_slots;
    uint32_t* ctrl;
    const int* uexp;
    const int* off;
    const int* order;      // MOE_MODE_ORDERED: position -> index into uexp/off, else null
    const int* pair;
    uint32_t* gu_done;
    // the gate/up sums a split publishes for the other: 8-byte words (float bits,
    // tag), [tile][split][pair][128]; a word is this launch's when its tag is
    unsigned long long* gu_part;
    uint32_t* gu_state;  // per (chunk, tile): bit s set once split s has published
    const uint8_t* x_mx;   // packed E2M1 terms of the block's rows (row T n + t) [rows][d/2], scales [rows][d/32]
    const uint8_t* x_sc;
    uint8_t* h_mx;         // packed E2M1 terms of the pairs' SwiGLU activations (row T P + t) [rows][f/2], scales
    uint8_t* h_sc;
    float* y_part;
    float* dbg_g;
    float* dbg_u;
};

// one stage: item, type, chunk id (work unit of <= CHUNK pairs of one expert), tile,
// split, stage index within the item, the item's stages, MMA N, scale buffer and
// row pitch, K base, activation rows, first activation row (down) / first pair
struct Meta {
    int item, type, c, blk, split, chunk, nchunks, nb, sbuf, sc, kbase, nrow, brow, p0, pad[2];
};

struct AccMeta {
    int item, type, c, blk, split, nb, p0, rc;
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

// instruction descriptor of kind::mxf4: E2M1 A and B (format code 1), fp32 D,
// K-major, M = 128, N = nb, E8M0 scales; with scale_vec::2X an MMA (K = 64) uses
// two scale bytes of each 32-bit scale word, starting at byte `sf` (0 or 2)
__device__ __forceinline__ uint32_t idesc(int nb, int sf) {
    return ((uint32_t)sf << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(nb >> 3) << 17) | (1u << 23) | (8u << 24) |
           ((uint32_t)sf << 29);
}

__device__ __forceinline__ void mma_mx(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id, uint32_t sfa, uint32_t sfb,
                                       bool acc) {
    asm volatile(
        "{ .reg .pred p; setp.ne.u32 p, %6, 0;\n"
        "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p; }" ::"r"(
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

// exchange slot of (accumulator row m, token n): rows of 16 floats, columns
// xor-swizzled by the row so that a warp reading one token's column hits
// distinct banks
__device__ __forceinline__ int xch_at(int m, int n) { return m * 16 + (n ^ (m & 15)); }

// item -> (type, chunk, tile, split).  Groups i = 0 .. V+lag-1 hold the gate/up
// items of chunk i (tile-major, splits adjacent; if i < V) followed by the down
// items of chunk i - lag (if that is a chunk), so a chunk's down items come lag
// chunks after its gate/up items.  Closed form over the three runs of group sizes.
__device__ void decode_item(const Params& p, int V, int item, int& type, int& v, int& blk, int& split) {
    const int n_gi = p.n_gu * S, n_dn = p.n_dn, lag = p.lag;
    split = 0;
    auto gu_at = [&](int g, int rest) {
        type = IT_GU;
        v = g;
        blk = rest / S;
        split = rest - blk * S;
    };
    auto dn_at = [&](int g, int rest) {
        type = IT_DN;
        v = g;
        blk = rest;
    };
    if (lag <= V) {
        const int a = lag * n_gi;                       // groups [0, lag): gate/up only
        if (item < a) return gu_at(item / n_gi, item % n_gi);
        const int w = n_gi + n_dn, b = a + (V - lag) * w;   // groups [lag, V): both
        if (item < b) {
            const int g = lag + (item - a) / w, rest = (item - a) % w;
            if (rest < n_gi) return gu_at(g, rest);
            return dn_at(g - lag, rest - n_gi);
        }
        const int g = V + (item - b) / n_dn;            // groups [V, V+lag): down only
        return dn_at(g - lag, (item - b) % n_dn);
    }
    const int a = V * n_gi;                             // groups [0, V): gate/up only
    if (item < a) return gu_at(item / n_gi, item % n_gi);
    return dn_at((item - a) / n_dn, (item - a) % n_dn);  // groups [lag, lag+V): down only
}

// the expert holding chunk c: the last u with cp[u] <= c
__device__ __forceinline__ int chunk_expert(const int* cp, int U, int c) {
    int lo = 0, hi = U - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cp[mid] <= c) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// bounded wait until (*flag & bits) != 0; false (with the timeout bit set) if it gave up
__device__ bool wait_bits(const Params& p, const uint32_t* flag, uint32_t bits) {
    if ((ld_acquire(flag) & bits) != 0u) return true;
    const uint64_t t0 = global_ns();
    while ((ld_acquire(flag) & bits) == 0u) {
        if (timed_out(p.ctrl)) return false;
        if (global_ns() - t0 > WAIT_LIMIT_NS) {
            set_error(p.ctrl, MOE_EBIT_TIMEOUT);
            return false;
        }
        __nanosleep(256);
    }
    return true;
}

// a claimed work item, decoded: its type, chunk, block, K split, slot and pairs
struct Plan {
    int item, type, cid, blk, split, z, p0, rc;
    int pv[CHUNK];  // gate/up items of blocks without a pair table in shared memory: the chunk's pairs
};

__device__ __forceinline__ void plan_item(const Params& p, int V, int U, const uint2* umeta, const int* cp, int item,
                                          int total, int ch, Plan& q) {
    q.item = item;
    if (item >= total) return;
    decode_item(p, V, item, q.type, q.cid, q.blk, q.split);
    const int u = chunk_expert(cp, U, q.cid);
    const uint2 mu = umeta[u];
    const int o0 = (int)(mu.y & 0xFFFFu), r = (int)(mu.y >> 16);
    q.z = (int)mu.x;
    q.p0 = o0 + ch * (q.cid - cp[u]);  // the chunk's first pair
    q.rc = min(ch, o0 + r - q.p0);     // and its pairs
}

// the chunk's pair entries (gate/up items gather the rows of their tokens); loaded
// one item ahead, written for the scale movers at the item's first stage
__device__ __forceinline__ void plan_pairs(const Params& p, int total, Plan& q) {
#pragma unroll
    for (int i = 0; i < CHUNK; i++) q.pv[i] = 0;
    if (q.item >= total || q.type != IT_GU) return;
#pragma unroll
    for (int i = 0; i < CHUNK; i++)
        if (i < q.rc) q.pv[i] = __ldcg(p.pair + q.p0 + i);
}

// bounded wait until *flag >= target; false (with the timeout bit set) if it gave up
__device__ bool wait_at_least(const Params& p, const uint32_t* flag, uint32_t target) {
    if (ld_acquire(flag) >= target) return true;
    const uint64_t t0 = global_ns();
    while (ld_acquire(flag) < target) {
        if (timed_out(p.ctrl)) return false;
        if (global_ns() - t0 > WAIT_LIMIT_NS) {
            set_error(p.ctrl, MOE_EBIT_TIMEOUT);
            return false;
        }
        __nanosleep(128);
    }
    return true;
}

// ---------------------------------------------------------------------------

template <int NBM>
__device__ void producer(const Params& p, int U, const uint2* umeta, const int* cp, unsigned char* smem,
                         unsigned char* scbuf, uint64_t* full, uint64_t* empty, uint64_t* mready, uint64_t* scf,
                         uint64_t* sce, Meta* meta, int first, uint16_t* tokb) {
    using C = Cfg<NBM>;
    tma_prefetch_desc(&p.a_gu);
    tma_prefetch_desc(&p.a_dn);
    tma_prefetch_desc(&p.s_gu);
    tma_prefetch_desc(&p.s_dn);
    const int V = cp[U];  // chunks
    const int total = V * (p.n_gu * S + p.n_dn);
    uint32_t stage = 0, phase = 0, pending = 0, pending_par = 0;
    uint32_t sc_any = 0u, sc_cnt = 0u;  // per scale buffer: armed at all, and the parity of its arm count
    bool ok = true;
    // Claims run two items ahead: the claim of the item after next goes out at the
    // first stage of the current item and is decoded one item later, so neither the
    // atomic's round trip nor the next item's dependency load (issued right after its
    // decoding) waits in line with the stages.
    Plan cur, nxt;
    plan_item(p, V, U, umeta, cp, first, total, C::CH, cur);
    if (tokb != nullptr) plan_pairs(p, total, cur);
    int claim_next = (int)atomicAdd(p.ctrl + CTRL_WORK_TC, 1u);
    uint32_t dep_cur = 0u;  // the current item's dependency word as last read
    if (cur.item < total) {
        if (p.slot_ready != nullptr) dep_cur = ld_acquire(p.slot_ready + cur.z);
        else if (cur.type != IT_GU) dep_cur = ld_acquire(p.gu_done + cur.cid);
    }
    for (int seq = 0; ok && cur.item < total; seq++) {
        const int item = cur.item, type = cur.type, cid = cur.cid, blk = cur.blk, split = cur.split;
        const int z = cur.z, p0 = cur.p0, rc = cur.rc;
        const bool gu = type == IT_GU;
        // gate/up items need the slot's gate/up planes (bit 0), down items its down planes (bit 1)
        if (p.slot_ready != nullptr && (dep_cur & (gu ? MOE_SLOT_GATE_UP : MOE_SLOT_DOWN)) == 0u)
            ok = wait_bits(p, p.slot_ready + z, gu ? MOE_SLOT_GATE_UP : MOE_SLOT_DOWN);
        if (ok && !gu && (p.slot_ready != nullptr || dep_cur < (uint32_t)p.n_gu)) {
            // the chunk's SwiGLU activations must be complete before the scale movers
            // read them (they read this item's stages only after its claim below)
            ok = wait_at_least(p, p.gu_done + cid, (uint32_t)p.n_gu);
        }
        if (!ok) break;
        const int kr = gu ? p.d / S : p.f;     // K range of the item
        const int kbase = gu ? split * kr : 0;
        const int nch = kr / KC;
        const int sc = kr / 32;                // scale bytes per row of the item
        const int nb = round16(T * rc);       // activation rows loaded = MMA N
        const int brow = T * p0;               // down: the chunk's rows of h
        const int row0 = gu ? blk * 64 : blk * 128;
        const int sbuf = seq & 1;
        unsigned char* sa = scbuf + sbuf * C::SCB;
        const uint32_t tx = (uint32_t)A_BYTES;
        const uint32_t tx_sc = (uint32_t)(128 * sc);
        int claim_after = total;
        uint32_t dep_nxt = 0u;
        nxt.item = total;
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
            mt.c = cid;
            mt.blk = blk;
            mt.split = split;
            mt.chunk = c;
            mt.nchunks = nch;
            mt.nb = nb;
            mt.sbuf = sbuf;
            mt.sc = sc;
            mt.kbase = kbase;
            mt.nrow = T * rc;
            mt.brow = brow;
            mt.p0 = p0;
            if (c == 0) {
                // the item's scales into its buffer, once the scale movers are done
                // with item seq-2, which used it last
                if (seq >= 2 && !mbar_wait(&sce[sbuf], (uint32_t)((seq >> 1) - 1) & 1u)) {
                    set_error(p.ctrl, MOE_EBIT_TIMEOUT);
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&scf[sbuf], tx_sc);
                if (gu && tokb != nullptr) {  // the chunk's tokens, read by the scale movers after the claim
#pragma unroll
                    for (int i = 0; i < CHUNK; i++)
                        if (i < rc) tokb[sbuf * CHUNK + i] = (uint16_t)(cur.pv[i] / p.k);
                }
                if (gu)
                    tma_load_4d(sa, &p.s_gu, &scf[sbuf], kbase / 32, row0, 0, z);
                else
                    tma_load_3d(sa, &p.s_dn, &scf[sbuf], 0, row0, z);
                sc_any |= 1u << sbuf;
                sc_cnt ^= 1u << sbuf;
            }
            // the stage is this item's now: the scale movers may prepare it while
            // its codes are in flight
            mbar_arrive(&mready[stage]);
            mbar_arrive_expect_tx(&full[stage], tx);
            unsigned char* st = smem + (size_t)stage * C::STAGE;
            const int kc = (kbase + c * KC) / 256;   // the stage's first 256-K piece
            if (gu)
                tma_load_5d(st, &p.a_gu, &full[stage], 0, row0, 0, kc, z);
            else
                tma_load_4d(st, &p.a_dn, &full[stage], 0, row0, kc, z);
            pending |= 1u << stage;
            pending_par = (pending_par & ~(1u << stage)) | (phase << stage);
            if (++stage == C::NST) {
                stage = 0;
                phase ^= 1u;
            }
            if (c == 0) {
                // the claim two items ahead, and the decoding of the next item (claimed
                // one item ago) with its dependency load, which lands during this item
                claim_after = (int)atomicAdd(p.ctrl + CTRL_WORK_TC, 1u);
                plan_item(p, V, U, umeta, cp, claim_next, total, C::CH, nxt);
                if (tokb != nullptr) plan_pairs(p, total, nxt);
                if (nxt.item < total) {
                    if (p.slot_ready != nullptr) dep_nxt = ld_acquire(p.slot_ready + nxt.z);
                    else if (nxt.type != IT_GU) dep_nxt = ld_acquire(p.gu_done + nxt.cid);
                }
            }
        }
        cur = nxt;
        claim_next = claim_after;
        dep_cur = dep_nxt;
    }
    // tell the consumers there is nothing more (after an error too, if a stage frees up)
    if (mbar_wait(&empty[stage], phase ^ 1u)) {
        pending &= ~(1u << stage);
        meta[stage].item = -1;
        mbar_arrive(&mready[stage]);
        mbar_arrive(&full[stage]);
    } else {
        set_error(p.ctrl, MOE_EBIT_TIMEOUT);
    }
    // no copy may still be in flight when the CTA exits
    for (int s = 0; s < C::NST; s++)
        if (pending & (1u << s)) mbar_wait(&full[s], (pending_par >> s) & 1u);
    for (int b = 0; b < 2; b++)
        if (sc_any & (1u << b)) mbar_wait(&scf[b], ((sc_cnt >> b) & 1u) ^ 1u);
}

// The activation operand of a stage (B) is copied by the four scale-mover warps
// straight from global memory into the stage's shared memory (16-byte cp.async,
// L2 only) as soon as the producer has claimed the stage, so the copies of every
// claimed stage are in flight at once and their latency hides behind the ring.
// Thread t copies 16-byte pieces j = t + 128 i (row j / (8 KCH), piece j % (8 KCH)
// of the row's KC/2 packed bytes) into the 128-byte-swizzled K-major layout the
// MMA reads (KCH regions of NBM rows of 128 bytes, piece cc of row r at
// 16 * (cc ^ (r % 8))).  Every warp also copies the stage's E8M0 scale bytes of
// activation rows lane, 32 + lane and 64 + lane into its own staging area, so
// each lane later reads only what it copied itself.
constexpr int BP = 8 * KCH;  // 16-byte pieces of a B row per stage

// source row of activation row `row` of a stage: gate/up gathers the E2M1 terms of
// the block rows of the chunk's pairs (T x the pair's token + term), down reads the
// chunk's rows of h (T x pair + term) in place.  tok: the block row of every pair
// (small blocks); else tokb, the block rows of the chunk's pairs (from the producer)
__device__ __forceinline__ int b_src_row(const Meta& m, int row, const uint16_t* tok, const uint16_t* tokb) {
    if (m.type != IT_GU) return m.brow + row;
    const int q = row / T;
    const int n = tok != nullptr ? (int)tok[m.p0 + q] : (int)tokb[m.sbuf * CHUNK + q];
    return T * n + (row - T * q);
}

// the source rows this thread copies for an item (data rows j / BP of its pieces
// j, scale rows lane, 32 + lane and 64 + lane), resolved once per item
template <int NBM>
struct BRows {
    int item = -1;
    int d[NBM * BP / Cfg<NBM>::MOV_T];
    int s[3];
};

// no memory clobber: the copy's destination is read only after cp_async_wait (which
// has one), so the compiler may keep everything else in registers around the copies
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src));
}

__device__ __forceinline__ void cp_async_wait(int pending) {
    switch (pending) {  // the oldest group of the thread is complete once at most `pending` remain
        case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
        case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
        case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
        case 3: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
        default: asm volatile("cp.async.wait_group 4;" ::: "memory"); break;
    }
}

// issue the copies of one claimed stage (one cp.async group per thread and stage)
// m is a copy in registers: the loop below reads its fields between the copies
template <int NBM>
__device__ __forceinline__ void b_issue(const Params& p, const Meta m, int t, int lane, uint32_t bst, uint32_t sbs,
                                        BRows<NBM>& r, const uint16_t* tok, const uint16_t* tokb) {
    using C = Cfg<NBM>;
    if (r.item != m.item) {
        r.item = m.item;
#pragma unroll
        for (int i = 0; i < NBM * BP / C::MOV_T; i++) {
            if (C::MOV_T * i >= m.nrow * BP) break;  // no row of this or later pieces is in use
            const int row = (t + C::MOV_T * i) / BP;
            r.d[i] = row < m.nrow ? b_src_row(m, row, tok, tokb) : 0;
        }
#pragma unroll
        for (int c = 0; c < 3; c++) {
            const int row = 32 * c + lane;
            r.s[c] = (row < m.nrow && row < NBM) ? b_src_row(m, row, tok, tokb) : 0;
        }
    }
    const bool gu = m.type == IT_GU;
    const uint8_t* src = gu ? p.x_mx : p.h_mx;
    const uint8_t* ssrc = gu ? p.x_sc : p.h_sc;
    const int ld = gu ? p.d : p.f;
    const int k0 = m.kbase + m.chunk * KC;
#pragma unroll
    for (int i = 0; i < NBM * BP / C::MOV_T; i++) {
        if (C::MOV_T * i >= m.nrow * BP) break;  // the same in the whole warp
        const int j = t + C::MOV_T * i, row = j / BP, c16 = j % BP, kh = c16 >> 3, cc = c16 & 7;
        if (row < m.nrow)
            cp_async16(bst + kh * (NBM * 128) + row * 128 + ((cc ^ (row & 7)) << 4),
                       src + (size_t)r.d[i] * (ld / 2) + k0 / 2 + c16 * 16);
    }
    static_assert(KC / 32 == 16, "one 16-byte scale copy per row and stage");
    if (t < 128) {  // the four scale warps
#pragma unroll
        for (int c = 0; c < 3; c++) {
            const int row = 32 * c + lane;
            if (row < m.nrow && row < NBM) cp_async16(sbs + row * 16, ssrc + (size_t)r.s[c] * (ld / 32) + k0 / 32);
        }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// the copy warps: per stage, the activation rows into the stage's B area (above);
// warps 2..5 also every E8M0 scale into tensor memory.  Scale of row m (A: weight row, B: activation
// row) for the stage's K blocks 4*set..4*set+3 is byte (kb % 4) of the 32-bit word
// at lane m % 32, column base + set*4 + m / 32; each warp writes the copy in its own
// lane quadrant.  Stages are finished in order: once the thread's copies of the
// oldest stage have landed (and, for an item's first stage, its A scales), the
// scales go to tensor memory and the warp releases the stage to the MMA.  After an
// item's last stage the warps release its scale buffer (sce).
template <int NBM>
__device__ void scale_mover(const Params& p, unsigned char* smem, unsigned char* scbuf, unsigned char* sbs_all,
                            uint32_t tbase, uint64_t* mready, uint64_t* scf, uint64_t* sce, uint64_t* sfr,
                            const Meta* meta, const uint16_t* tok, const uint16_t* tokb) {
    using C = Cfg<NBM>;
    const int lane = threadIdx.x & 31, q = (threadIdx.x >> 5) & 3, t = threadIdx.x - 64;
    const bool scw = t < 128;  // warps 2..5 also move the scales (warp w writes lane quadrant w % 4)
    const uint32_t sbs = smem_u32(sbs_all) + (uint32_t)(q * C::NST * NBM * 16);  // this warp's scale staging
    uint32_t is = 0, iph = 0;   // next stage to issue, and the parity of its claim
    uint32_t fs = 0;            // next stage to finish
    int inflight = 0;
    bool ended = false, ok = true;
    uint32_t scph = 0;          // parity of the next phase of each A-scale buffer
    BRows<NBM> rows;
    while (ok) {
        // every claimed stage goes out, up to the whole ring
        while (!ended && inflight < C::NST) {
            bool claimed;
            if (inflight == 0) {
                claimed = __shfl_sync(0xffffffffu, mbar_wait(&mready[is], iph) ? 1 : 0, 0) != 0;
                if (!claimed) {
                    if (lane == 0) set_error(p.ctrl, MOE_EBIT_TIMEOUT);
                    ok = false;
                    break;
                }
            } else {
                claimed = __all_sync(0xffffffffu, mbar_peek(&mready[is], iph));
                if (!claimed) break;
            }
            const Meta& m = meta[is];
            if (m.item < 0) {
                ended = true;
                break;
            }
            b_issue<NBM>(p, m, t, lane, smem_u32(smem + (size_t)is * C::STAGE + A_BYTES), sbs + is * (NBM * 16),
                         rows, tok, tokb);
            inflight++;
            if (++is == (uint32_t)C::NST) {
                is = 0;
                iph ^= 1u;
            }
        }
        if (!ok || inflight == 0) break;
        // finish the oldest stage
        const Meta m = meta[fs];
        cp_async_wait(inflight - 1);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the copies, for the MMA's reads
        if (!scw) {  // a copy-only warp: the stage's copies of this warp have landed
            __syncwarp();
            if (lane == 0) mbar_arrive(&sfr[fs]);
            inflight--;
            if (++fs == (uint32_t)C::NST) fs = 0;
            continue;
        }
        if (m.chunk == 0) {  // the item's A scales have landed
            if (__shfl_sync(0xffffffffu, mbar_wait(&scf[m.sbuf], (scph >> m.sbuf) & 1u) ? 1 : 0, 0) == 0) {
                if (lane == 0) set_error(p.ctrl, MOE_EBIT_TIMEOUT);
                ok = false;
                break;
            }
            scph ^= 1u << m.sbuf;
        }
        const uint32_t sa = smem_u32(scbuf + m.sbuf * C::SCB);
        const uint32_t sb = sbs + fs * (NBM * 16);
        uint4 bs[3];
#pragma unroll
        for (int c = 0; c < 3; c++) {
            const int row = 32 * c + lane;
            bs[c] = (row < m.nrow && row < NBM) ? lds128(sb + row * 16) : make_uint4(0, 0, 0, 0);
        }
        const int kb_off = m.chunk * (KC / 32);
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
#pragma unroll
        for (int set = 0; set < KC / 128; set++) {
            uint32_t wa[4];
#pragma unroll
            for (int c = 0; c < 4; c++) wa[c] = lds32(sa + (32 * c + lane) * m.sc + kb_off + 4 * set);
            const uint32_t w0 = set == 0 ? bs[0].x : set == 1 ? bs[0].y : set == 2 ? bs[0].z : bs[0].w;
            const uint32_t w1 = set == 0 ? bs[1].x : set == 1 ? bs[1].y : set == 2 ? bs[1].z : bs[1].w;
            const uint32_t w2 = set == 0 ? bs[2].x : set == 1 ? bs[2].y : set == 2 ? bs[2].z : bs[2].w;
            tm_st4(tbase + C::TM_SFA + fs * SF_COLS + set * 4 + lane_base, wa[0], wa[1], wa[2], wa[3]);
            tm_st4(tbase + C::TM_SFB + fs * SF_COLS + set * 4 + lane_base, w0, w1, w2, 0u);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        fence_before();
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&sfr[fs]);
            if (m.chunk == m.nchunks - 1) mbar_arrive(&sce[m.sbuf]);  // done reading the item's scales
        }
        inflight--;
        if (++fs == (uint32_t)C::NST) fs = 0;
    }
    // no copy may still be in flight when the CTA exits
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// warp 1, one thread: four MMAs (K = 64 each) per stage into the item's accumulator
template <int NBM>
__device__ void mma_issuer(const Params& p, unsigned char* smem, uint32_t tbase, uint64_t* full, uint64_t* empty,
                           uint64_t* sfr, uint64_t* acc_full, uint64_t* acc_empty, uint64_t* done, const Meta* meta,
                           AccMeta* am) {
    using C = Cfg<NBM>;
    uint32_t stage = 0, phase = 0, it = 0;
    bool ok = true;
    while (true) {
        if (!mbar_wait(&full[stage], phase)) {
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
            a.c = m.c;
            a.blk = m.blk;
            a.split = m.split;
            a.nb = m.nb;
            a.p0 = m.p0;
            a.rc = m.nrow / T;
        }
        const uint32_t st = smem_u32(smem + (size_t)stage * C::STAGE);
#pragma unroll
        for (int ks = 0; ks < KC / 64; ks++) {
            // K = 64 packed codes = 32 bytes of a 128-byte row piece; four MMAs per piece
            const int kh = ks >> 2;
            const uint64_t ad = sdesc(st + kh * 16384 + (ks & 3) * 32);
            const uint64_t bd = sdesc(st + A_BYTES + kh * (NBM * 128) + (ks & 3) * 32);
            mma_mx(tbase + b * C::ACC_SET + (ks % C::NACC) * C::ACC_COLS, ad, bd, idesc(m.nb, (ks & 1) * 2),
                   tbase + C::TM_SFA + stage * SF_COLS + (ks >> 1) * 4,
                   tbase + C::TM_SFB + stage * SF_COLS + (ks >> 1) * 4, m.chunk != 0 || ks >= C::NACC);
        }
        mma_commit(&empty[stage]);
        if (m.chunk == m.nchunks - 1) {
            mbar_arrive(&acc_full[b]);  // publishes am[b] (release)
            mma_commit(&acc_full[b]);   // completes when the accumulator is final
            it++;
        }
        if (++stage == C::NST) {
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

// A partial sum with the tag of the launch that wrote it: one 8-byte word, written
// and read whole, so a reader that sees the tag sees the value stored with it.
__device__ __forceinline__ unsigned long long tagged(float v, uint32_t tag) {
    return ((unsigned long long)tag << 32) | __float_as_uint(v);
}

// The gate and up sums of one output row from another split: each word is read
// from L2 until it carries this launch's tag (bounded: after the wait limit, or once
// any wait of the launch has given up, the timeout bit is set and the words are
// taken as they are).
__device__ __forceinline__ void tagged_pair(const Params& p, const unsigned long long* pg,
                                            const unsigned long long* pu, uint32_t tag, float& g, float& u) {
    unsigned long long wg = __ldcg(pg), wu = __ldcg(pu);
    if ((uint32_t)(wg >> 32) != tag || (uint32_t)(wu >> 32) != tag) {
        const uint64_t t0 = global_ns();
        while (true) {
            __nanosleep(64);
            if ((uint32_t)(wg >> 32) != tag) wg = __ldcg(pg);
            if ((uint32_t)(wu >> 32) != tag) wu = __ldcg(pu);
            if ((uint32_t)(wg >> 32) == tag && (uint32_t)(wu >> 32) == tag) break;
            if (timed_out(p.ctrl)) break;
            if (global_ns() - t0 > WAIT_LIMIT_NS) {
                set_error(p.ctrl, MOE_EBIT_TIMEOUT);
                break;
            }
        }
    }
    g = __uint_as_float((uint32_t)wg);
    u = __uint_as_float((uint32_t)wu);
}

// the last four warps: TMEM lane quadrant q = warp % 4, accumulator row m = 32q + lane
template <int NBM>
__device__ void epilogue(const Params& p, uint32_t tbase, float* xch, uint32_t tag, uint64_t* acc_full,
                         uint64_t* acc_empty, const AccMeta* am) {
    using C = Cfg<NBM>;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, q = warp & 3, ew = warp - Cfg<NBM>::EPI_W0;
    const int N = p.n_rows;
    __shared__ int s_flag;  // the epilogue warps' shared decision of the current gate/up item
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
        // The item's result, read 16 columns at a time up to the MMA's width: each
        // column is its accumulators summed in order (0 + acc0 + acc1), and each pair's
        // T term columns are summed in order into ps[pair].  Columns are visited in
        // order, so a pair whose columns straddle two 16-column pieces carries on.
        float ps[NBM / T];
        const uint32_t ta0 = tbase + b * C::ACC_SET + ((uint32_t)(32 * q) << 16);
#pragma unroll
        for (int h = 0; h < NBM / 16; h++) {
            if (h > 0 && a.nb <= 16 * h) break;  // the MMA wrote nb columns (same in the whole warp)
            uint32_t w[C::NACC][16];
#pragma unroll
            for (int ai = 0; ai < C::NACC; ai++) tm_ld16(ta0 + ai * C::ACC_COLS + 16 * h, w[ai]);
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
            for (int i = 0; i < 16; i++) {
                const int col = 16 * h + i, n = col / T, tt = col - (col / T) * T;
                if (n < NBM / T) {
                    float v = 0.f;
#pragma unroll
                    for (int ai = 0; ai < C::NACC; ai++) v += __uint_as_float(w[ai][i]);
                    ps[n] = tt == 0 ? v : ps[n] + v;
                }
            }
        }
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[b]);
        const int m = 32 * q + lane;
        const int o0 = a.p0, r = a.rc;  // the chunk's pairs: o0 .. o0 + r - 1, MMA columns T per pair
        if (a.type == IT_GU) {
            // each pair's sum over its T term columns; rows 0..63 gate, 64..127 up
#pragma unroll
            for (int n = 0; n < NBM / T; n++)
                if (n < r) xch[xch_at(m, n)] = ps[n];
            if (ew == 0 && lane == 0) s_flag = 1;
            epi_sync();
            // The two splits of a tile meet here; exactly one of them adds the sums:
            //  - split 1 reads split 0's words first; if they all carry this launch's
            //    tag it combines at once, with no atomic;
            //  - otherwise a split publishes its own sums as tagged words and sets its
            //    bit in the tile's state word (split 0 always does); the one that finds
            //    the other's bit already set combines.
            // Either way the sums are added in split order, so the result does not
            // depend on which split combined.
            const int j0 = a.blk * 64;
            const size_t tile_base = (size_t)a.blk * S * p.nk;
            const unsigned long long* osrc = p.gu_part + (tile_base + (size_t)(1 - a.split) * p.nk + o0) * 128;
            float og[2] = {0.f, 0.f}, ou[2] = {0.f, 0.f};  // the other split's sums of this thread's first two tasks
            bool have = a.split == 1;
            if (a.split == 1) {
#pragma unroll
                for (int q2 = 0; q2 < 2; q2++) {
                    const int task = ew + 4 * q2;
                    if (task < 2 * r) {
                        const int col = task >> 1, jrow = 32 * (task & 1) + lane;
                        const unsigned long long wg = __ldcg(osrc + (size_t)col * 128 + jrow);
                        const unsigned long long wu = __ldcg(osrc + (size_t)col * 128 + 64 + jrow);
                        have = have && (uint32_t)(wg >> 32) == tag && (uint32_t)(wu >> 32) == tag;
                        og[q2] = __uint_as_float((uint32_t)wg);
                        ou[q2] = __uint_as_float((uint32_t)wu);
                    }
                }
                if (!have) s_flag = 0;
                epi_sync();
            }
            int combine = a.split == 1 ? s_flag : 0;
            if (!combine) {
                // publish: part[tile][split][pair][128], one tagged word per sum (the
                // reader checks every word's tag, so no fence is needed)
                for (int task = ew; task < 2 * r; task += 4) {
                    const int col = task >> 1, half = task & 1;
                    const int row = 64 * half + lane;
                    unsigned long long* dst = p.gu_part + (tile_base + (size_t)a.split * p.nk + o0 + col) * 128;
                    dst[row] = tagged(xch[xch_at(row, col)], tag);
                    dst[row + 32] = tagged(xch[xch_at(row + 32, col)], tag);
                }
                epi_sync();
                if (ew == 0 && lane == 0) {
                    const uint32_t mine = 1u << a.split;
                    s_flag = (atomicOr(p.gu_state + (size_t)a.c * p.n_gu + a.blk, mine) & (3u ^ mine)) != 0u;
                }
                epi_sync();
                combine = s_flag;
                have = false;  // the other split's words are read again below
            }
            if (combine) {
                bool wrote = false;
                for (int task = ew, q2 = 0; task < 2 * r; task += 4, q2++) {
                    const int col = task >> 1, jb = task & 1;
                    const int P = o0 + col;
                    const int j = 32 * jb + lane;
                    float go, uo;
                    if (have && q2 < 2) {
                        go = q2 == 0 ? og[0] : og[1];
                        uo = q2 == 0 ? ou[0] : ou[1];
                    } else {
                        tagged_pair(p, osrc + (size_t)col * 128 + j, osrc + (size_t)col * 128 + 64 + j, tag, go, uo);
                    }
                    const float gm = xch[xch_at(j, col)], um = xch[xch_at(64 + j, col)];
                    float g = 0.f, u = 0.f;  // split 0's sums, then split 1's
                    g += a.split == 0 ? gm : go;
                    u += a.split == 0 ? um : uo;
                    g += a.split == 0 ? go : gm;
                    u += a.split == 0 ? uo : um;
                    const float hv = g / (1.f + expf(-g)) * u;
                    if (p.debug) {
                        const size_t o = (size_t)(p.n_shared * N + P) * p.f + j0 + j;
                        p.dbg_g[o] = g;
                        p.dbg_u[o] = u;
                    }
                    uint32_t qv[T], sbits[T];
                    mx_split(hv, qv, sbits);
#pragma unroll
                    for (int t = 0; t < T; t++) {
                        store_e2m1_block(p.h_mx + (size_t)(T * P + t) * (p.f / 2) + (j0 + 32 * jb) / 2, qv[t]);
                        if (lane == 0) p.h_sc[(size_t)(T * P + t) * (p.f / 32) + (j0 >> 5) + jb] = (uint8_t)sbits[t];
                    }
                    wrote = true;
                }
                if (wrote) __threadfence();
                epi_sync();  // also: every read of xch and s_flag is done before the next item
                if (ew == 0 && lane == 0) red_release_add(p.gu_done + a.c, 1u);
            } else {
                epi_sync();  // every read of xch and s_flag is done before the next item
            }
        } else {
            const int m0 = a.blk * 128;
            int pid[NBM / T];  // the chunk's pair ids, all loaded before the first store
#pragma unroll
            for (int col = 0; col < NBM / T; col++) pid[col] = col < r ? __ldcg(p.pair + o0 + col) : 0;
#pragma unroll
            for (int col = 0; col < NBM / T; col++)
                if (col < r) p.y_part[(size_t)pid[col] * p.d + m0 + m] = ps[col];
        }
        it++;
    }
}

template <int NBM>
__global__ void __launch_bounds__(Cfg<NBM>::NTHREADS, 1) tc_expert_kernel(const __grid_constant__ Params p) {
    using C = Cfg<NBM>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    unsigned char* scbuf = smem + (size_t)C::NST * C::STAGE;
    unsigned char* sbs = scbuf + 2 * C::SCB;
    float* xch = reinterpret_cast<float*>(sbs + C::SBS_BYTES);
    uint2* umeta = reinterpret_cast<uint2*>(xch + XCH_FLOATS);
    int* cp = reinterpret_cast<int*>(umeta + C::MAX_U);  // [MAX_U + 1] chunk prefix
    uint16_t* tok = C::TOKS > 0 ? reinterpret_cast<uint16_t*>(cp + C::MAX_U + 1) : nullptr;  // [TOKS]
    uint16_t* tokb = reinterpret_cast<uint16_t*>(cp + C::MAX_U + 1) + C::TOKS;              // [2][CHUNK]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)C::NST * C::STAGE + 2 * C::SCB + C::SBS_BYTES +
                                                 XCH_FLOATS * 4 + ((C::META_BYTES + 15) & ~15));
    uint64_t* full = bars;
    uint64_t* empty = full + C::NST;
    uint64_t* sfr = empty + C::NST;
    uint64_t* mready = sfr + C::NST;
    uint64_t* scf = mready + C::NST;
    uint64_t* sce = scf + 2;
    uint64_t* acc_full = sce + 2;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* done = acc_empty + 2;
    Meta* meta = reinterpret_cast<Meta*>(done + 1);
    AccMeta* am = reinterpret_cast<AccMeta*>(meta + C::NST);
    static_assert((4 * C::NST + 9) * 8 + C::NST * sizeof(Meta) + 2 * sizeof(AccMeta) + 8 <= 1024, "barrier area");
    uint32_t* tslot = reinterpret_cast<uint32_t*>(am + 2);
    __shared__ int s_last;

    const int tid = threadIdx.x, warp = tid >> 5;
    if (tid == 0) tl_begin(p.ctrl, TL_ROUTED);
    if (tid == 0) {
        for (int s = 0; s < C::NST; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&sfr[s], C::NMOV);
            mbar_init(&mready[s], 1);
        }
        mbar_init(&scf[0], 1);
        mbar_init(&scf[1], 1);
        mbar_init(&sce[0], 4);
        mbar_init(&sce[1], 4);
        for (int b = 0; b < 2; b++) {
            mbar_init(&acc_full[b], 2);
            mbar_init(&acc_empty[b], 4);
        }
        mbar_init(done, 1);
        mbar_fence_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                     "r"(C::TM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    // the set-up above overlaps the previous kernel on the stream; everything below
    // reads the routing's results.  Directly after the shared experts that ran beside
    // the routing, this CTA only starts once a CTA of theirs has triggered its
    // dependents, which each does only after the routing has completed: no wait here
    // (the acquire below drops stale L1 lines), and the wait for the shared experts
    // is at the end.
    if (!p.after_shared) griddep_wait();
    griddep_launch_dependents();
    __shared__ int s_u;
    __shared__ uint32_t s_tag;
    // the producer's first claim goes out now: its latency overlaps the loads below
    int first = 0;
    if (tid == 0) {
        s_u = (int)ld_acquire(p.ctrl + CTRL_UNIQUE);
        // this launch's tag: one more than the launches before it on this workspace
        // (never 0, the value of a zeroed workspace)
        s_tag = __ldcg(p.ctrl + CTRL_EPOCH_TC) + 1u;
        first = (int)atomicAdd(p.ctrl + CTRL_WORK_TC, 1u);
    }
    __syncthreads();
    const int U = min(s_u, C::MAX_U);
    // every expert's slot and pair range (all loads in flight at once), then the
    // prefix of its chunk counts (one warp: contiguous runs per lane, then a scan)
    for (int u = tid; u < U; u += C::NTHREADS) {
        const int ui = ordered_index(p.order, u, U);
        int z = __ldg(p.expert_slot + __ldcg(p.uexp + ui));
        const int o0 = __ldcg(p.off + ui), r = __ldcg(p.off + ui + 1) - o0;
        if (z < 0 || z >= p.n_slots) {
            set_error(p.ctrl, MOE_EBIT_BAD_SLOT);
            z = 0;
        }
        umeta[u] = make_uint2((uint32_t)z, (uint32_t)o0 | ((uint32_t)r << 16));
    }
    if (tok != nullptr)  // the block row of every pair (small blocks only)
        for (int i = tid; i < p.nk && i < C::TOKS; i += C::NTHREADS) tok[i] = (uint16_t)(__ldcg(p.pair + i) / p.k);
    __syncthreads();
    if (warp == 1) {
        const int lane = tid & 31, per = (U + 31) / 32, b0 = lane * per, b1 = min(U, b0 + per);
        int sum = 0;
        for (int u = b0; u < b1; u++) sum += ((int)(umeta[u].y >> 16) + C::CH - 1) / C::CH;
        int incl = sum;
        for (int o = 1; o < 32; o <<= 1) {
            const int up = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += up;
        }
        int run = incl - sum;
        for (int u = b0; u < b1; u++) {
            cp[u] = run;
            run += ((int)(umeta[u].y >> 16) + C::CH - 1) / C::CH;
        }
        if (lane == 31) cp[U] = incl;
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tbase = *tslot;

    if (warp == 0) {
        if ((tid & 31) == 0)
            producer<NBM>(p, U, umeta, cp, smem, scbuf, full, empty, mready, scf, sce, meta, first,
                          tok != nullptr ? nullptr : tokb);
    } else if (warp == 1) {
        if ((tid & 31) == 0) mma_issuer<NBM>(p, smem, tbase, full, empty, sfr, acc_full, acc_empty, done, meta, am);
    } else if (warp < C::EPI_W0) {
        scale_mover<NBM>(p, smem, scbuf, sbs, tbase, mready, scf, sce, sfr, meta, tok, tokb);
    } else {
        epilogue<NBM>(p, tbase, xch, s_tag, acc_full, acc_empty, am);
    }

    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(C::TM_COLS));
    // the last CTA to finish leaves the counters clean for the next call
    if (tid == 0) {
        __threadfence();
        s_last = atomicAdd(p.ctrl + CTRL_EXIT_TC, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (s_last) {
        __threadfence();
        const int V = cp[U];
        for (int i = tid; i < V; i += C::NTHREADS) p.gu_done[i] = 0;
        for (int i = tid; i < V * p.n_gu; i += C::NTHREADS) p.gu_state[i] = 0;
        if (tid == 0) {
            p.ctrl[CTRL_WORK_TC] = 0;
            p.ctrl[CTRL_EXIT_TC] = 0;
            p.ctrl[CTRL_EPOCH_TC] = s_tag;  // the next launch tags with s_tag + 1
        }
    }
    if (tid == 0) tl_end(p.ctrl, TL_ROUTED);
    if (p.after_shared && tid == 0) griddep_wait();  // complete only after the shared experts
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
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &qr) ==
                cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(ptr);
        return static_cast<EncodeTiledFn>(nullptr);
    }();
    return fn;
}

// tiled map of rank 3 to 5: dims[0] contiguous, byte strides of dims 1..rank-1
static bool map_nd(CUtensorMap* m, CUtensorMapDataType type, const void* addr, int rank, const uint64_t* dims,
                   const uint64_t* strides, const uint32_t* box, bool swizzle) {
    EncodeTiledFn enc = encode_fn();
    if (!enc || rank < 3 || rank > 5) return false;
    cuuint64_t gd[5], gs[4];
    cuuint32_t bx[5], es[5] = {1, 1, 1, 1, 1};
    for (int i = 0; i < rank; i++) {
        gd[i] = dims[i];
        bx[i] = box[i];
    }
    for (int i = 0; i + 1 < rank; i++) gs[i] = strides[i];
    return enc(m, type, (cuuint32_t)rank, const_cast<void*>(addr), gd, gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NBM>
static int launch(const Params& p, cudaStream_t stream) {
    using C = Cfg<NBM>;
    static const cudaError_t attr = kernel_smem_attrs(tc_expert_kernel<NBM>, (int)C::SMEM);
    if (attr != cudaSuccess) return MOE_ERR_CUDA;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return MOE_ERR_CUDA;
    if (launch_chained(tc_expert_kernel<NBM>, dim3(sms), dim3(C::NTHREADS), C::SMEM, stream, p) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

}  // namespace tc

// Shapes the block-scaled path serves: gate/up K splits that are whole stages
// (multiples of 256 elements) with a scale row that fits the per-item buffer, a
// down K range of whole stages (scale row likewise), 64-row gate/up and 128-row
// down tiles.
bool tc_expert_supported(int d, int f, int n_rows) {
    using namespace tc;
    return d % (KC * S) == 0 && d % 128 == 0 && d / S / 32 <= SC_MAX && f % KC == 0 && f % 64 == 0 &&
           f / 32 <= SC_MAX && n_rows >= 1;
}

int tc_expert_launch(const moe_desc* desc, int n_rows, int mode, const moe_pool* routed, const int32_t* expert_slot,
                     const uint32_t* slot_ready, int n_shared, void* ws, int n_rows_max, float* y_part,
                     cudaStream_t stream) {
    using namespace tc;
    const int d = desc->d_model, f = desc->d_ff, E = desc->n_experts, k = desc->top_k;
    // first pair and pair count share one 32-bit word per expert; blocks of up to 16
    // rows with at most 256 pairs run the 32-column configuration, in chunks of up
    // to 6 pairs (a row's arithmetic is the same in both configurations)
    const bool small = n_rows <= 16 && n_rows * k <= Cfg<32>::TOKS;
    if (n_rows * k >= 65536 || E > Cfg<80>::MAX_U) return MOE_ERR_UNSUPPORTED;
    const WsLayout L = ws_layout(d, f, E, k, n_rows_max, n_shared);
    char* base = static_cast<char*>(ws);
    thread_local Params p;  // filled per call, copied into the launch
    memset(&p, 0, sizeof(p));
    // slab planes: [gate codes | gate scales | up codes | up scales | down codes | down scales]
    const char* pool = static_cast<const char*>(routed->base);
    const uint64_t per = (uint64_t)f * d / 2 + (uint64_t)f * (d / 32);  // one gate or up matrix with its scales
    const uint64_t slot = (uint64_t)routed->slot_bytes, ns = (uint64_t)routed->n_slots;
    const char* down_c = pool + 2 * per;
    const char* down_s = down_c + (uint64_t)d * f / 2;
    const CUtensorMapDataType U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    {   // 256-K pieces of a code row are 128 bytes apart; a box is 64 gate + 64 up rows x KCH pieces
        const uint64_t dims[5] = {128, (uint64_t)f, 2, (uint64_t)d / 256, ns};
        const uint64_t str[4] = {(uint64_t)d / 2, per, 128, slot};
        const uint32_t box[5] = {128, 64, 2, KCH, 1};
        if (!map_nd(&p.a_gu, U8, pool, 5, dims, str, box, true)) return MOE_ERR_UNSUPPORTED;
    }
    {
        const uint64_t dims[4] = {(uint64_t)d / 32, (uint64_t)f, 2, ns}, str[3] = {(uint64_t)d / 32, per, slot};
        const uint32_t box[4] = {(uint32_t)(d / S / 32), 64, 2, 1};
        if (!map_nd(&p.s_gu, U8, pool + (uint64_t)f * d / 2, 4, dims, str, box, false)) return MOE_ERR_UNSUPPORTED;
    }
    {
        const uint64_t dims[4] = {128, (uint64_t)d, (uint64_t)f / 256, ns}, str[3] = {(uint64_t)f / 2, 128, slot};
        const uint32_t box[4] = {128, 128, KCH, 1};
        if (!map_nd(&p.a_dn, U8, down_c, 4, dims, str, box, true)) return MOE_ERR_UNSUPPORTED;
    }
    {
        const uint64_t dims[3] = {(uint64_t)f / 32, (uint64_t)d, ns}, str[2] = {(uint64_t)f / 32, slot};
        const uint32_t box[3] = {(uint32_t)(f / 32), 128, 1};
        if (!map_nd(&p.s_dn, U8, down_s, 3, dims, str, box, false)) return MOE_ERR_UNSUPPORTED;
    }
    p.d = d;
    p.f = f;
    p.k = k;
    p.n_rows = n_rows;
    p.n_shared = n_shared;
    p.nk = n_rows * k;
    p.n_gu = f / 64;
    p.n_dn = d / 128;
    p.lag = 1 << 30;  // every gate/up item before the first down item
    p.debug = (mode & MOE_MODE_DEBUG_GU) ? 1 : 0;
    p.after_shared = (mode & MOE_MODE_AFTER_SHARED) ? 1 : 0;

    p.expert_slot = expert_slot;
    p.slot_ready = slot_ready;
    p.n_slots = routed->n_slots;
    p.ctrl = reinterpret_cast<uint32_t*>(base + L.ctrl);
    p.uexp = reinterpret_cast<const int*>(base + L.uexp);
    p.off = reinterpret_cast<const int*>(base + L.off);
    p.order = (mode & MOE_MODE_ORDERED) ? reinterpret_cast<const int*>(base + L.uorder) : nullptr;
    p.pair = reinterpret_cast<const int*>(base + L.pair);
    p.gu_done = reinterpret_cast<uint32_t*>(base + L.gu_done_tc);
    p.gu_part = reinterpret_cast<unsigned long long*>(base + L.gu_part);
    p.gu_state = reinterpret_cast<uint32_t*>(base + L.gu_state);
    p.x_mx = reinterpret_cast<const uint8_t*>(base + L.x_mx);
    p.x_sc = reinterpret_cast<const uint8_t*>(base + L.x_sc);
    p.h_mx = reinterpret_cast<uint8_t*>(base + L.h_mx);
    p.h_sc = reinterpret_cast<uint8_t*>(base + L.h_sc);
    p.y_part = y_part;
    p.dbg_g = reinterpret_cast<float*>(base + L.dbg_g);
    p.dbg_u = reinterpret_cast<float*>(base + L.dbg_u);
    // a chunk holds at most 6 (small blocks) or 16 pairs, T MMA columns each
    return small ? launch<32>(p, stream) : launch<80>(p, stream);
}

}  // namespace moe
