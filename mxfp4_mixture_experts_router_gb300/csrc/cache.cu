// Device expert cache: a slab pool in HBM whose slots hold (layer, expert)
// slabs, filled from a pinned host pool on upload streams.
//
// Pages: "Run Kimi 3.1 locally on one GPU", section "One GPU, three storage
// tiers": experts that do not fit in device memory are streamed in as the router
// asks for them, and compute on an expert starts as its data lands.  Here the
// lower tier is pinned host memory (the NVMe tier is out of scope).
//
// Host side only.  A request names the experts one layer of a block needs; hits
// keep their slot, misses take a free slot or evict one: plain LRU, or "keep the
// experts used by two rows or more": the least recently used slot whose last
// block used it on a single row, and when every candidate was used by several
// rows, the most recently used of them (so a working set larger than the cache
// keeps the longer-held experts instead of cycling through all of them).
// For the misses, in this order:
//   compute stream: each victim's ready flag is written 0 (after every earlier
//                   kernel on that stream, so after every reader of the old slab)
//   compute stream: an event is recorded
//   upload stream (one of n, round robin): waits for the event, copies the
//                   slab's gate+up part, sets MOE_SLOT_GATE_UP, copies the down
//                   part, sets MOE_SLOT_READY (both bits)
// The expert kernels wait (bounded) for the bit each work item needs, so the
// gate/up work on an expert starts while its down part is still in flight.
// With zero upload streams the cache only plans (slot assignment and misses,
// no CUDA calls): the policy logic runs the same way without a GPU.
#include "common.cuh"

#include <chrono>
#include <list>
#include <new>
#include <thread>
#include <unordered_map>
#include <vector>

typedef CUresult (*WriteValue32Fn)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);


__global__ void cache_flag_kernel(uint32_t* flag, uint32_t value) { *flag = value; }

struct moe_cache {
    char* base = nullptr;
    int64_t slot_bytes = 0, slab_bytes = 0, gu_bytes = 0;
    int32_t n_slots = 0;
    uint32_t* ready = nullptr;
    int policy = MOE_CACHE_LRU;
    std::vector<cudaStream_t> streams;
    std::vector<cudaEvent_t> events;
    int ev_next = 0;
    WriteValue32Fn write_value = nullptr;

    struct Slot {
        uint64_t key = 0;
        bool used = false;
        int64_t last = -1;      // request that last used the slot
        int32_t rows = 0;       // rows of that request's block that used it
        std::list<int32_t>::iterator pos;
    };
    std::vector<Slot> slots;
    std::list<int32_t> order;   // front: most recently used
    std::vector<int32_t> free_slots;
    std::unordered_map<uint64_t, int32_t> where;
    int64_t seq = 0;
    moe_cache_stats stats = {};
};

namespace {

uint64_t cache_key(int32_t layer, int32_t expert) { return ((uint64_t)(uint32_t)layer << 32) | (uint32_t)expert; }

void touch(moe_cache* c, int32_t s) {
    moe_cache::Slot& sl = c->slots[s];
    if (sl.used) c->order.erase(sl.pos);
    c->order.push_front(s);
    sl.pos = c->order.begin();
}

// a slot for a miss of request `seq`, never one this request uses: a free one;
// else under MOE_CACHE_LRU the least recently used; under
// MOE_CACHE_KEEP_MULTI_ROW the least recently used single-row slot, and failing
// that the most recently used slot
int32_t pick_victim(moe_cache* c, int64_t seq) {
    if (!c->free_slots.empty()) {
        const int32_t s = c->free_slots.back();
        c->free_slots.pop_back();
        return s;
    }
    if (c->policy == MOE_CACHE_KEEP_MULTI_ROW) {
        for (auto it = c->order.rbegin(); it != c->order.rend(); ++it) {
            const moe_cache::Slot& sl = c->slots[*it];
            if (sl.last != seq && sl.rows < 2) return *it;
        }
        for (auto it = c->order.begin(); it != c->order.end(); ++it)
            if (c->slots[*it].last != seq) return *it;
        return -1;
    }
    for (auto it = c->order.rbegin(); it != c->order.rend(); ++it)
        if (c->slots[*it].last != seq) return *it;
    return -1;
}

int write_flag(moe_cache* c, cudaStream_t s, uint32_t* flag, uint32_t value) {
    if (c->write_value) {
        return c->write_value(reinterpret_cast<CUstream>(s), reinterpret_cast<CUdeviceptr>(flag), value, 0) ==
                       CUDA_SUCCESS
                   ? MOE_OK
                   : MOE_ERR_CUDA;
    }
    cache_flag_kernel<<<1, 1, 0, s>>>(flag, value);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// A host function on an upload stream that returns once (*flag & bits) != 0: the
// stream's next copy then reads a chunk the lower tier has finished writing.  The
// wait is bounded (10 s), so the stream always moves on; the GPU itself never waits
// on host memory.
struct HostWait {
    const uint32_t* flag;
    uint32_t bits;
};

void CUDART_CB host_wait(void* arg) {
    HostWait* w = static_cast<HostWait*>(arg);
    const auto t0 = std::chrono::steady_clock::now();
    while ((__atomic_load_n(w->flag, __ATOMIC_ACQUIRE) & w->bits) == 0u) {
        if (std::chrono::steady_clock::now() - t0 > std::chrono::seconds(10)) break;
        std::this_thread::yield();
    }
    delete w;
}

int enqueue_host_wait(cudaStream_t s, const uint32_t* flag, uint32_t bits) {
    HostWait* w = new (std::nothrow) HostWait{flag, bits};
    if (!w) return MOE_ERR_CUDA;
    if (cudaLaunchHostFunc(s, host_wait, w) != cudaSuccess) {
        delete w;
        return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

void release(moe_cache* c) {
    for (cudaStream_t s : c->streams) {
        cudaStreamSynchronize(s);
        cudaStreamDestroy(s);
    }
    for (cudaEvent_t e : c->events) cudaEventDestroy(e);
    delete c;
}

}  // namespace

extern "C" int moe_cache_create(const moe_desc* desc, void* slot_base, int64_t slot_bytes, int32_t n_slots,
                                uint32_t* slot_ready, int32_t n_streams, int32_t policy, moe_cache** out) {
    if (!desc || !out || n_slots < 1 || n_streams < 0 || n_streams > 64) return MOE_ERR_INVALID_ARG;
    if (policy != MOE_CACHE_LRU && policy != MOE_CACHE_KEEP_MULTI_ROW) return MOE_ERR_INVALID_ARG;
    *out = nullptr;
    const int64_t slab = (int64_t)moe_slab_bytes(desc, MOE_FMT_MXFP4);
    if (slab <= 0 || slot_bytes < slab) return MOE_ERR_INVALID_ARG;
    if (n_streams > 0 && (!slot_base || !slot_ready)) return MOE_ERR_INVALID_ARG;
    moe_cache* c = new (std::nothrow) moe_cache();
    if (!c) return MOE_ERR_INVALID_ARG;
    const int64_t d = desc->d_model, f = desc->d_ff;
    c->base = static_cast<char*>(slot_base);
    c->slot_bytes = slot_bytes;
    c->slab_bytes = slab;
    c->gu_bytes = 2 * (f * d / 2 + f * (d / 32));  // [gate codes | gate scales | up codes | up scales]
    c->n_slots = n_slots;
    c->ready = slot_ready;
    c->policy = policy;
    c->slots.resize(n_slots);
    for (int32_t s = n_slots - 1; s >= 0; s--) c->free_slots.push_back(s);
    if (n_streams > 0) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuStreamWriteValue32", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            c->write_value = reinterpret_cast<WriteValue32Fn>(fn);

        for (int i = 0; i < n_streams; i++) {
            cudaStream_t s;
            if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) {
                release(c);
                return MOE_ERR_CUDA;
            }
            c->streams.push_back(s);
        }
        for (int i = 0; i < 8; i++) {
            cudaEvent_t e;
            if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
                release(c);
                return MOE_ERR_CUDA;
            }
            c->events.push_back(e);
        }
        // every slot starts empty
        if (cudaMemset(slot_ready, 0, sizeof(uint32_t) * (size_t)n_slots) != cudaSuccess) {
            release(c);
            return MOE_ERR_CUDA;
        }
    }
    *out = c;
    return MOE_OK;
}

static int cache_request(moe_cache* c, int32_t layer, int32_t count, const int32_t* experts, const int32_t* rows,
                         const void* const* host_src, const uint32_t* const* host_ready, int32_t* slot_out,
                         int32_t* miss_out, void* compute_stream) {
    if (!c || count < 0 || (count > 0 && (!experts || !slot_out))) return MOE_ERR_INVALID_ARG;
    if (count > c->n_slots) return MOE_ERR_UNSUPPORTED;
    const bool gpu = !c->streams.empty();
    if (gpu && count > 0 && !host_src) return MOE_ERR_INVALID_ARG;
    const int64_t seq = ++c->seq;
    c->stats.requests++;
    // hits first, so that no expert of this request is evicted for another one
    std::vector<int32_t> miss_idx;
    for (int32_t i = 0; i < count; i++) {
        const uint64_t key = cache_key(layer, experts[i]);
        auto it = c->where.find(key);
        const int32_t r = rows ? rows[i] : 1;
        if (it != c->where.end()) {
            const int32_t s = it->second;
            touch(c, s);
            c->slots[s].last = seq;
            c->slots[s].rows = r;
            c->slots[s].used = true;
            slot_out[i] = s;
            if (miss_out) miss_out[i] = 0;
            c->stats.hits++;
        } else {
            miss_idx.push_back(i);
        }
    }
    std::vector<int32_t> victims;
    for (int32_t i : miss_idx) {
        const int32_t s = pick_victim(c, seq);
        if (s < 0) return MOE_ERR_UNSUPPORTED;  // cannot happen while count <= n_slots
        moe_cache::Slot& sl = c->slots[s];
        if (sl.used) {
            c->where.erase(sl.key);
            c->stats.evictions++;
        }
        sl.key = cache_key(layer, experts[i]);
        touch(c, s);
        sl.used = true;
        sl.last = seq;
        sl.rows = rows ? rows[i] : 1;
        c->where[sl.key] = s;
        slot_out[i] = s;
        if (miss_out) miss_out[i] = 1;
        c->stats.misses++;
        c->stats.bytes_uploaded += c->slab_bytes;
        victims.push_back(s);
    }
    if (!gpu || victims.empty()) return MOE_OK;

    cudaStream_t cs = static_cast<cudaStream_t>(compute_stream);
    for (int32_t s : victims)
        if (write_flag(c, cs, c->ready + s, 0u) != MOE_OK) return MOE_ERR_CUDA;
    cudaEvent_t ev = c->events[c->ev_next];
    c->ev_next = (c->ev_next + 1) % (int)c->events.size();
    if (cudaEventRecord(ev, cs) != cudaSuccess) return MOE_ERR_CUDA;
    const int ns = (int)c->streams.size();
    const int used_streams = (int)victims.size() < ns ? (int)victims.size() : ns;
    for (int k = 0; k < used_streams; k++)
        if (cudaStreamWaitEvent(c->streams[k], ev, 0) != cudaSuccess) return MOE_ERR_CUDA;
    for (size_t m = 0; m < victims.size(); m++) {
        const int32_t s = victims[m];
        const int32_t i = miss_idx[m];
        cudaStream_t us = c->streams[m % ns];
        char* dst = c->base + (size_t)s * (size_t)c->slot_bytes;
        const char* src = static_cast<const char*>(host_src[i]);
        if (!src) return MOE_ERR_INVALID_ARG;
        const uint32_t* hr = host_ready ? host_ready[i] : nullptr;
        // a slab still being read into host memory: each chunk waits for its bit
        if (hr && enqueue_host_wait(us, hr, MOE_SLOT_GATE_UP) != MOE_OK) return MOE_ERR_CUDA;
        if (cudaMemcpyAsync(dst, src, (size_t)c->gu_bytes, cudaMemcpyHostToDevice, us) != cudaSuccess)
            return MOE_ERR_CUDA;
        if (write_flag(c, us, c->ready + s, MOE_SLOT_GATE_UP) != MOE_OK) return MOE_ERR_CUDA;
        if (hr && enqueue_host_wait(us, hr, MOE_SLOT_DOWN) != MOE_OK) return MOE_ERR_CUDA;
        if (cudaMemcpyAsync(dst + c->gu_bytes, src + c->gu_bytes, (size_t)(c->slab_bytes - c->gu_bytes),
                            cudaMemcpyHostToDevice, us) != cudaSuccess)
            return MOE_ERR_CUDA;
        if (write_flag(c, us, c->ready + s, MOE_SLOT_READY) != MOE_OK) return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

extern "C" int moe_cache_request(moe_cache* c, int32_t layer, int32_t count, const int32_t* experts,
                                 const int32_t* rows, const void* const* host_src, int32_t* slot_out,
                                 int32_t* miss_out, void* compute_stream) {
    return cache_request(c, layer, count, experts, rows, host_src, nullptr, slot_out, miss_out, compute_stream);
}

extern "C" int moe_cache_request_staged(moe_cache* c, int32_t layer, int32_t count, const int32_t* experts,
                                        const int32_t* rows, const void* const* host_src,
                                        const uint32_t* const* host_ready, int32_t* slot_out, int32_t* miss_out,
                                        void* compute_stream) {
    if (count > 0 && !host_ready) return MOE_ERR_INVALID_ARG;
    return cache_request(c, layer, count, experts, rows, host_src, host_ready, slot_out, miss_out, compute_stream);
}

extern "C" int moe_cache_lookup(const moe_cache* c, int32_t layer, int32_t count, const int32_t* experts,
                                int32_t* resident_out) {
    if (!c || count < 0 || (count > 0 && (!experts || !resident_out))) return MOE_ERR_INVALID_ARG;
    for (int32_t i = 0; i < count; i++) resident_out[i] = c->where.count(cache_key(layer, experts[i])) ? 1 : 0;
    return MOE_OK;
}

extern "C" int moe_cache_stats_get(const moe_cache* c, moe_cache_stats* out) {
    if (!c || !out) return MOE_ERR_INVALID_ARG;
    *out = c->stats;
    return MOE_OK;
}

extern "C" int moe_cache_sync(moe_cache* c) {
    if (!c) return MOE_ERR_INVALID_ARG;
    for (cudaStream_t s : c->streams)
        if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
}

extern "C" int moe_cache_destroy(moe_cache* c) {
    if (!c) return MOE_ERR_INVALID_ARG;
    release(c);
    return MOE_OK;
}
