// Step a12: a page pool held in pinned host memory.
//
// papernotes.org "IceCache: Memory-Efficient KV-cache Management for
// Long-Sequence LLMs", 关键设计 4: the selected pages are scattered in host
// memory, so they are first collected into one contiguous host staging
// buffer and moved to the GPU in a single high-throughput transfer, instead
// of many small copies; IceCache popular-science article
// (aitangshan.cn/news/751385), section 四: everything needed is gathered into
// one staging area and sent in one transfer.
//
// The pool is pinned and mapped into the device address space, so it serves
// two ways:
//   - staged: host worker threads copy the selected pages (ids read back by
//     the caller) into a pinned staging buffer laid out as the contiguous
//     kbuf | vbuf | buf_len, then one cudaMemcpyAsync moves it to the device;
//   - direct: its device-visible pointers go into ice_index.pool_k / pool_v,
//     and the build and decode kernels write and read the pages over the
//     CPU-GPU link (NVLink-C2C on GB300) with no host copy and no host sync.
#include <condition_variable>
#include <cstring>
#include <functional>
#include <mutex>
#include <thread>
#include <vector>

#include "common.cuh"
#include "internal.h"

struct ice_host_pool {
    void *k_host = nullptr, *v_host = nullptr;  // pinned, mapped
    void *k_dev = nullptr, *v_dev = nullptr;    // device-visible aliases
    size_t pool_bytes = 0;
    void *staging = nullptr;  // pinned
    size_t staging_bytes = 0;
    cudaEvent_t copied = nullptr;  // the last staged transfer has read the staging buffer
    bool pending = false;
    // worker threads
    std::vector<std::thread> workers;
    std::mutex mu;
    std::condition_variable cv_work, cv_done;
    std::function<void(int)> job;
    int generation = 0, remaining = 0;
    bool stop = false;
};

namespace ice {
namespace {

void worker_loop(ice_host_pool *hp, int id) {
    int seen = 0;
    for (;;) {
        std::function<void(int)> job;
        {
            std::unique_lock<std::mutex> lk(hp->mu);
            hp->cv_work.wait(lk, [&] { return hp->stop || hp->generation != seen; });
            if (hp->stop) return;
            seen = hp->generation;
            job = hp->job;
        }
        job(id);
        {
            std::lock_guard<std::mutex> lk(hp->mu);
            if (--hp->remaining == 0) hp->cv_done.notify_all();
        }
    }
}

// Runs fn(worker) on every worker thread and waits for all of them.
void run_all(ice_host_pool *hp, std::function<void(int)> fn) {
    std::unique_lock<std::mutex> lk(hp->mu);
    hp->job = std::move(fn);
    hp->remaining = (int)hp->workers.size();
    ++hp->generation;
    hp->cv_work.notify_all();
    hp->cv_done.wait(lk, [&] { return hp->remaining == 0; });
}

void release(ice_host_pool *hp) {
    if (!hp) return;
    {
        std::lock_guard<std::mutex> lk(hp->mu);
        hp->stop = true;
    }
    hp->cv_work.notify_all();
    for (auto &t : hp->workers)
        if (t.joinable()) t.join();
    if (hp->copied) {
        cudaEventSynchronize(hp->copied);
        cudaEventDestroy(hp->copied);
    }
    if (hp->k_host) cudaFreeHost(hp->k_host);
    if (hp->v_host) cudaFreeHost(hp->v_host);
    if (hp->staging) cudaFreeHost(hp->staging);
    delete hp;
}

}  // namespace
}  // namespace ice

using namespace ice;

extern "C" {

ice_status ice_host_pool_create(size_t pool_bytes, size_t staging_bytes, int32_t n_threads, ice_host_pool **out) {
    if (!out || pool_bytes == 0 || n_threads < 1 || n_threads > 256) return ICE_ERR_INVALID_ARG;
    *out = nullptr;
    ice_host_pool *hp = new ice_host_pool();
    hp->pool_bytes = pool_bytes;
    hp->staging_bytes = staging_bytes;
    const unsigned flags = cudaHostAllocMapped | cudaHostAllocPortable;
    if (fault_armed("alloc") || cudaHostAlloc(&hp->k_host, pool_bytes, flags) != cudaSuccess ||
        cudaHostAlloc(&hp->v_host, pool_bytes, flags) != cudaSuccess ||
        (staging_bytes && cudaHostAlloc(&hp->staging, staging_bytes, cudaHostAllocPortable) != cudaSuccess)) {
        cudaGetLastError();
        release(hp);
        return ICE_ERR_OOM;
    }
    if (fault_armed("hostpool") || cudaHostGetDevicePointer(&hp->k_dev, hp->k_host, 0) != cudaSuccess ||
        cudaHostGetDevicePointer(&hp->v_dev, hp->v_host, 0) != cudaSuccess ||
        cudaEventCreateWithFlags(&hp->copied, cudaEventDisableTiming) != cudaSuccess) {
        cudaGetLastError();
        release(hp);
        return ICE_ERR_CUDA;
    }
    for (int i = 0; i < n_threads; ++i) hp->workers.emplace_back(worker_loop, hp, i);
    *out = hp;
    return ICE_OK;
}

ice_status ice_host_pool_destroy(ice_host_pool *hp) {
    if (!hp) return ICE_ERR_INVALID_ARG;
    release(hp);
    return ICE_OK;
}

ice_status ice_host_pool_pointers(const ice_host_pool *hp, void **pool_k_dev, void **pool_v_dev, void **pool_k_host,
                                  void **pool_v_host) {
    if (!hp) return ICE_ERR_INVALID_ARG;
    if (pool_k_dev) *pool_k_dev = hp->k_dev;
    if (pool_v_dev) *pool_v_dev = hp->v_dev;
    if (pool_k_host) *pool_k_host = hp->k_host;
    if (pool_v_host) *pool_v_host = hp->v_host;
    return ICE_OK;
}

size_t ice_host_pool_staging_bytes(const ice_params *p, int32_t max_sel) {
    if (!p || max_sel < 1) return 0;
    const size_t U = (size_t)p->batch * p->n_kv_heads;
    const size_t esz = p->dtype == ICE_BF16 ? 2 : 4;
    const size_t page = (size_t)p->page_size * p->head_dim * esz;
    return 2 * U * max_sel * page + U * max_sel * sizeof(int32_t);
}

ice_status ice_host_pool_gather_h2d(ice_host_pool *hp, const ice_params *p, const int32_t *sel_pages_host,
                                    const int32_t *sel_count_host, const int32_t *page_len_host, int32_t max_sel,
                                    void *dst_dev, size_t dst_bytes, void *stream) {
    if (!hp || !p || !sel_pages_host || !sel_count_host || !page_len_host || !dst_dev || max_sel < 1)
        return ICE_ERR_INVALID_ARG;
    if (p->head_dim != kHeadDim || p->page_size != kPage || (p->dtype != ICE_BF16 && p->dtype != ICE_FP32))
        return ICE_ERR_UNSUPPORTED;
    const size_t need = ice_host_pool_staging_bytes(p, max_sel);
    if (need > hp->staging_bytes || need > dst_bytes) return ICE_ERR_CAPACITY;
    const size_t U = (size_t)p->batch * p->n_kv_heads;
    const size_t esz = p->dtype == ICE_BF16 ? 2 : 4;
    const size_t page = (size_t)kPage * kHeadDim * esz;
    if ((size_t)p->page_cap * page * U > hp->pool_bytes) return ICE_ERR_CAPACITY;
    // the previous staged transfer must have finished reading the staging buffer
    if (hp->pending && cudaEventSynchronize(hp->copied) != cudaSuccess) return ICE_ERR_CUDA;
    char *kb = static_cast<char *>(hp->staging);
    char *vb = kb + U * max_sel * page;
    int32_t *bl = reinterpret_cast<int32_t *>(vb + U * max_sel * page);
    const char *pk = static_cast<const char *>(hp->k_host);
    const char *pv = static_cast<const char *>(hp->v_host);
    const int nt = (int)hp->workers.size();
    bool bad = false;
    std::mutex bad_mu;
    run_all(hp, [&](int w) {
        for (size_t u = w; u < U; u += nt) {
            const int n = sel_count_host[u];
            if (n < 0 || n > max_sel) {  // a count the selection cannot have produced
                std::lock_guard<std::mutex> lk(bad_mu);
                bad = true;
                continue;
            }
            for (int x = 0; x < max_sel; ++x) {
                const size_t slot = u * max_sel + x;
                if (x >= n) {
                    bl[slot] = 0;
                    continue;
                }
                const int pg = sel_pages_host[slot];
                if (pg < 0 || pg >= p->page_cap) {
                    std::lock_guard<std::mutex> lk(bad_mu);
                    bad = true;
                    bl[slot] = 0;
                    continue;
                }
                const size_t src = (u * p->page_cap + pg) * page;
                std::memcpy(kb + slot * page, pk + src, page);
                std::memcpy(vb + slot * page, pv + src, page);
                bl[slot] = page_len_host[u * p->page_cap + pg];
            }
        }
    });
    if (bad) return ICE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the one bulk transfer of this layer
    if (fault_armed("copy") || cudaMemcpyAsync(dst_dev, hp->staging, need, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaEventRecord(hp->copied, s) != cudaSuccess) {
        cudaGetLastError();
        return ICE_ERR_CUDA;
    }
    hp->pending = true;
    return ICE_OK;
}

}  // extern "C"
