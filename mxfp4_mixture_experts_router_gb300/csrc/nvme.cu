// NVMe expert tier: expert slabs read from files (one file per drive, each drive
// holding a replica of the same slabs) into pinned host memory, from where the
// device expert cache uploads them.
//
// Pages: "Run Kimi 3.1 locally on one GPU", section "Read the experts the router
// needs": the experts live on several NVMe drives (a RAID0 set, a second drive,
// an external one); reads go straight to pinned memory (O_DIRECT), each read goes
// to the replica that is expected to finish it first, every drive has its own cap
// on reads in flight, and a decode fill comes in two chunks (gate+up first, so
// compute on an expert can start before its down part has arrived).
//
// Host only.  A replica is a file and a queue served by `depth` reader threads
// (the drive's concurrency cap).  A read is placed on the replica whose pending
// bytes plus the read's own, divided by the replica's measured bandwidth (an
// exponentially weighted average of its completed reads), is smallest.  A read
// fills [0, first) of the slab, sets MOE_SLOT_GATE_UP in the caller's flag, then
// fills the rest and sets MOE_SLOT_READY.  A failed read still sets its bits, with
// MOE_NVME_FAILED added, so that nothing waiting on the flag waits forever.
#include <fcntl.h>
#include <sys/stat.h>
#include <unistd.h>

#include <atomic>
#include <chrono>
#include <condition_variable>
#include <cstring>
#include <deque>
#include <mutex>
#include <new>
#include <string>
#include <thread>
#include <vector>

#include "common.cuh"

namespace {

struct Read {
    int32_t body;
    char* dst;
    int64_t first;
    volatile uint32_t* flag;
};

struct Replica {
    std::string path;
    int fd_direct = -1;   // O_DIRECT descriptor (or -1)
    int fd_buffered = -1;
    std::deque<Read> q;
    int64_t pending = 0;  // bytes queued or in flight
    double bw = 2e9;      // bytes per second, measured
    int64_t bytes = 0, reads = 0, failures = 0;
    double busy_s = 0;
};

int64_t now_ns() {
    return std::chrono::duration_cast<std::chrono::nanoseconds>(std::chrono::steady_clock::now().time_since_epoch())
        .count();
}

}  // namespace

struct moe_nvme {
    int64_t slab_bytes = 0, stride = 0;
    int32_t n_bodies = 0;
    std::vector<Replica> reps;
    std::vector<std::thread> threads;
    std::mutex m;
    std::condition_variable cv;
    bool stop = false;
};

namespace {

constexpr int64_t ALIGN = 4096;

// reads [off, off + len) of body b's slab into dst + off; O_DIRECT when every
// address and size is aligned, else the buffered descriptor
bool read_range(Replica& r, int64_t file_off, char* dst, int64_t len) {
    const bool direct = r.fd_direct >= 0 && (file_off % ALIGN) == 0 && ((uintptr_t)dst % ALIGN) == 0 &&
                        (len % ALIGN) == 0;
    const int fd = direct ? r.fd_direct : r.fd_buffered;
    int64_t done = 0;
    while (done < len) {
        const ssize_t got = pread(fd, dst + done, (size_t)(len - done), (off_t)(file_off + done));
        if (got <= 0) return false;
        done += got;
    }
    return true;
}

void serve(moe_nvme* s, int ri) {
    Replica& r = s->reps[ri];
    while (true) {
        Read rd;
        {
            std::unique_lock<std::mutex> lk(s->m);
            s->cv.wait(lk, [&] { return s->stop || !r.q.empty(); });
            if (r.q.empty()) return;
            rd = r.q.front();
            r.q.pop_front();
        }
        const int64_t t0 = now_ns();
        const int64_t base = (int64_t)rd.body * s->stride;
        bool ok = read_range(r, base, rd.dst, rd.first);
        __atomic_fetch_or(const_cast<uint32_t*>(rd.flag), MOE_SLOT_GATE_UP | (ok ? 0u : MOE_NVME_FAILED),
                          __ATOMIC_RELEASE);
        const bool ok2 = read_range(r, base + rd.first, rd.dst + rd.first, s->slab_bytes - rd.first);
        __atomic_fetch_or(const_cast<uint32_t*>(rd.flag), MOE_SLOT_READY | (ok2 ? 0u : MOE_NVME_FAILED),
                          __ATOMIC_RELEASE);
        const double dt = (now_ns() - t0) * 1e-9;
        std::lock_guard<std::mutex> lk(s->m);
        r.pending -= s->slab_bytes;
        r.reads++;
        r.bytes += s->slab_bytes;
        r.busy_s += dt;
        if (!(ok && ok2)) r.failures++;
        if (dt > 0) r.bw = 0.8 * r.bw + 0.2 * (s->slab_bytes / dt);
    }
}

void shutdown(moe_nvme* s) {
    {
        std::lock_guard<std::mutex> lk(s->m);
        s->stop = true;
    }
    s->cv.notify_all();
    for (std::thread& t : s->threads)
        if (t.joinable()) t.join();
    for (Replica& r : s->reps) {
        if (r.fd_direct >= 0) close(r.fd_direct);
        if (r.fd_buffered >= 0) close(r.fd_buffered);
    }
    delete s;
}

}  // namespace

extern "C" int moe_nvme_open(const char* const* paths, int32_t n_replicas, int64_t slab_bytes, int64_t slab_stride,
                             int32_t n_bodies, int32_t depth, moe_nvme** out) {
    if (!paths || !out || n_replicas < 1 || n_replicas > 16 || slab_bytes <= 0 || slab_stride < slab_bytes ||
        n_bodies < 1 || depth < 1 || depth > 64)
        return MOE_ERR_INVALID_ARG;
    *out = nullptr;
    moe_nvme* s = new (std::nothrow) moe_nvme();
    if (!s) return MOE_ERR_INVALID_ARG;
    s->slab_bytes = slab_bytes;
    s->stride = slab_stride;
    s->n_bodies = n_bodies;
    s->reps.resize(n_replicas);
    for (int i = 0; i < n_replicas; i++) {
        Replica& r = s->reps[i];
        if (!paths[i]) {
            shutdown(s);
            return MOE_ERR_INVALID_ARG;
        }
        r.path = paths[i];
        r.fd_buffered = open(paths[i], O_RDONLY);
        if (r.fd_buffered < 0) {
            shutdown(s);
            return MOE_ERR_INVALID_ARG;
        }
        struct stat st;
        if (fstat(r.fd_buffered, &st) != 0 || st.st_size < (off_t)((n_bodies - 1) * slab_stride + slab_bytes)) {
            shutdown(s);
            return MOE_ERR_INVALID_ARG;
        }
#ifdef O_DIRECT
        r.fd_direct = open(paths[i], O_RDONLY | O_DIRECT);  // -1 where the file system refuses it
#endif
    }
    for (int i = 0; i < n_replicas; i++)
        for (int t = 0; t < depth; t++) s->threads.emplace_back(serve, s, i);
    *out = s;
    return MOE_OK;
}

extern "C" int moe_nvme_read(moe_nvme* s, int32_t body, void* dst, int64_t first_bytes, volatile uint32_t* flag,
                             int32_t* replica_out) {
    if (!s || !dst || !flag || body < 0 || body >= s->n_bodies || first_bytes < 0 || first_bytes > s->slab_bytes)
        return MOE_ERR_INVALID_ARG;
    *flag = 0u;
    std::lock_guard<std::mutex> lk(s->m);
    // the replica expected to finish this read first
    int best = 0;
    double best_t = 1e300;
    for (int i = 0; i < (int)s->reps.size(); i++) {
        const Replica& r = s->reps[i];
        const double t = (double)(r.pending + s->slab_bytes) / r.bw;
        if (t < best_t) {
            best_t = t;
            best = i;
        }
    }
    Replica& r = s->reps[best];
    r.q.push_back(Read{body, static_cast<char*>(dst), first_bytes, flag});
    r.pending += s->slab_bytes;
    if (replica_out) *replica_out = best;
    s->cv.notify_all();
    return MOE_OK;
}

extern "C" int moe_nvme_wait(const volatile uint32_t* flag, uint32_t bits, int64_t timeout_ns) {
    if (!flag) return MOE_ERR_INVALID_ARG;
    const int64_t t0 = now_ns();
    while ((__atomic_load_n(const_cast<const uint32_t*>(flag), __ATOMIC_ACQUIRE) & bits) != bits) {
        if (now_ns() - t0 > timeout_ns) return MOE_ERR_TIMEOUT;
        std::this_thread::yield();
    }
    return (*flag & MOE_NVME_FAILED) ? MOE_ERR_IO : MOE_OK;
}

extern "C" int moe_nvme_stats_get(moe_nvme* s, int32_t replica, moe_nvme_stats* out) {
    if (!s || !out || replica < 0 || replica >= (int)s->reps.size()) return MOE_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(s->m);
    const Replica& r = s->reps[replica];
    out->reads = r.reads;
    out->bytes = r.bytes;
    out->failures = r.failures;
    out->pending_bytes = r.pending;
    out->bandwidth = r.bw;
    out->busy_seconds = r.busy_s;
    out->direct = r.fd_direct >= 0 ? 1 : 0;
    return MOE_OK;
}

extern "C" int moe_nvme_close(moe_nvme* s) {
    if (!s) return MOE_ERR_INVALID_ARG;
    shutdown(s);
    return MOE_OK;
}
