/*
 * fvif_hostmem.cu -- page-locked host buffers for fvif_score_host.
 *
 * fvif_score_host copies each chunk of host frames to the device with the
 * copy engine.  How fast that copy runs depends on how the host buffer was
 * made.  Measured on a GB300 with a Grace host, 8 GB buffers from
 * cudaHostAlloc copied at rates that varied from run to run and step to
 * step (from 211 GB/s down to 23 GB/s within one process, while a freshly
 * allocated 1 GiB buffer ran at 211 GB/s), whereas anonymous memory aligned
 * to the transparent-huge-page size, advised for huge pages and then
 * registered with cudaHostRegister ran at 210.7 GB/s in every trial.  These
 * two functions make buffers of the second kind, so callers can stage
 * their frames where the host path moves them fastest.
 */
#include <sys/mman.h>

#include <cstdint>
#include <cstdio>
#include <mutex>
#include <unordered_map>

#include "../../include/fvif.h"
#include "fvif_internal.h"

namespace {

std::mutex g_host_mutex;
std::unordered_map<void *, std::pair<void *, size_t>> g_host; /* -> map */

/* Alignment of the buffers: the transparent-huge-page size when the
 * kernel reports one (2 MiB on 4 KiB-page kernels, 512 MiB on 64 KiB-page
 * ones), at least 2 MiB, at most 1 GiB. */
size_t huge_page_bytes()
{
    static const size_t bytes = [] {
        size_t v = 0;
        if (FILE *f = std::fopen(
                "/sys/kernel/mm/transparent_hugepage/hpage_pmd_size", "r")) {
            unsigned long long u = 0;
            if (std::fscanf(f, "%llu", &u) == 1)
                v = (size_t)u;
            std::fclose(f);
        }
        const size_t lo = (size_t)2 << 20, hi = (size_t)1 << 30;
        if (v < lo || v > hi || (v & (v - 1)) != 0)
            v = lo;
        return v;
    }();
    return bytes;
}

} // namespace

extern "C" void *fvif_host_alloc(size_t bytes)
{
    if (bytes == 0)
        return nullptr;
    /* the start is aligned to the huge-page size; the length is rounded
     * only to 2 MiB, so a small request does not pin a whole huge page of
     * the larger sizes some kernels use */
    const size_t align = huge_page_bytes();
    const size_t gran = (size_t)2 << 20;
    const size_t size = (bytes + gran - 1) / gran * gran;
    if (size < bytes || size + align < size)
        return nullptr;
    /* map align bytes more than needed, then keep the aligned part */
    void *raw = mmap(nullptr, size + align, PROT_READ | PROT_WRITE,
                     MAP_PRIVATE | MAP_ANONYMOUS, -1, 0);
    if (raw == MAP_FAILED)
        return nullptr;
    const uintptr_t r = reinterpret_cast<uintptr_t>(raw);
    const uintptr_t a = (r + align - 1) & ~(uintptr_t)(align - 1);
    if (a > r)
        munmap(raw, a - r);
    if (r + align > a)
        munmap(reinterpret_cast<void *>(a + size), r + align - a);
    void *p = reinterpret_cast<void *>(a);
    madvise(p, size, MADV_HUGEPAGE); /* advice only: ignored if refused */
    if (cudaHostRegister(p, size, cudaHostRegisterPortable) != cudaSuccess) {
        cudaGetLastError();
        munmap(p, size);
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_host_mutex);
    g_host[p] = std::make_pair(p, size);
    return p;
}

extern "C" void fvif_host_free(void *p)
{
    if (!p)
        return;
    size_t size = 0;
    {
        std::lock_guard<std::mutex> lock(g_host_mutex);
        auto it = g_host.find(p);
        if (it == g_host.end())
            return;
        size = it->second.second;
        g_host.erase(it);
    }
    cudaHostUnregister(p);
    munmap(p, size);
}
