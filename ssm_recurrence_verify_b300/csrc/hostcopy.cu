// libssmverify: host -> device copies driven by the SMs.
//
// The host front end (ssm_recurrence_verify_b300/hostpipe.py) moves every
// step's draft-token inputs from page-locked host memory to the device. On
// B300 machines the copy engines move host -> device at 12-14 GB/s for the
// megabyte-sized transfers of a step, while the SMs reading the same page-
// locked memory through its unified device address reach 35-37 GB/s. This
// kernel does that: each thread moves 16-byte vectors, the grid strided over
// the transfer.

#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <stdint.h>

#include "ssmverify.h"
#include "ssm_internal.h"

namespace {

constexpr int kPullThreads = 512;

__global__ void __launch_bounds__(kPullThreads) ssm_pull_kernel(uint4 *dst, const uint4 *src, long long nvec,
                                                                 unsigned char *dtail, const unsigned char *stail,
                                                                 int ntail) {
    const long long stride = (long long)gridDim.x * kPullThreads;
    for (long long i = blockIdx.x * (long long)kPullThreads + threadIdx.x; i < nvec; i += stride) dst[i] = src[i];
    if (blockIdx.x == 0 && (int)threadIdx.x < ntail) dtail[threadIdx.x] = stail[threadIdx.x];
}

// Several 16-byte aligned copies in one grid: vector i of the concatenation
// belongs to the segment whose running start it passes; each segment's last
// bytes % 16 bytes are copied by block 0.
struct PullSegs {
    uint4 *dst[SSM_COPY_MAX_SEGMENTS];
    const uint4 *src[SSM_COPY_MAX_SEGMENTS];
    long long end[SSM_COPY_MAX_SEGMENTS];  // running end of each segment, in vectors
    int tail[SSM_COPY_MAX_SEGMENTS];       // bytes past the segment's last whole vector
    int n;
};

__global__ void __launch_bounds__(kPullThreads) ssm_pull_segments_kernel(const PullSegs sg) {
    const long long total = sg.end[sg.n - 1];
    const long long stride = (long long)gridDim.x * kPullThreads;
    for (long long i = blockIdx.x * (long long)kPullThreads + threadIdx.x; i < total; i += stride) {
        int k = 0;
        while (i >= sg.end[k]) ++k;  // n <= 8 segments
        const long long j = i - (k > 0 ? sg.end[k - 1] : 0);
        sg.dst[k][j] = sg.src[k][j];
    }
    if (blockIdx.x == 0) {
        for (int k = 0; k < sg.n; ++k) {
            const long long nv = sg.end[k] - (k > 0 ? sg.end[k - 1] : 0);
            if ((int)threadIdx.x < sg.tail[k])
                reinterpret_cast<unsigned char *>(sg.dst[k] + nv)[threadIdx.x] =
                    reinterpret_cast<const unsigned char *>(sg.src[k] + nv)[threadIdx.x];
        }
    }
}

__global__ void __launch_bounds__(kPullThreads) ssm_pull_bytes_kernel(unsigned char *dst, const unsigned char *src,
                                                                       long long n) {
    const long long stride = (long long)gridDim.x * kPullThreads;
    for (long long i = blockIdx.x * (long long)kPullThreads + threadIdx.x; i < n; i += stride) dst[i] = src[i];
}

bool is_host_locked(const void *p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();  // clear the sticky error of an unknown pointer
        return false;
    }
    return at.type == cudaMemoryTypeHost;
}

bool is_device(const void *p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

int sm_count() {
    static std::atomic<int> cache{0};
    int v = cache.load(std::memory_order_relaxed);
    if (v == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) !=
                                                      cudaSuccess)
            return 148;
        cache.store(v, std::memory_order_relaxed);
    }
    return v;
}

}  // namespace

extern "C" {

int ssm_copy_from_host(void *dst, const void *src, int64_t bytes, void *stream) {
    if (bytes < 0) return SSM_ERR_SHAPE;
    if (bytes == 0) return SSM_OK;
    if (dst == nullptr || src == nullptr) return SSM_ERR_NULL;
    const uintptr_t s = reinterpret_cast<uintptr_t>(src), d = reinterpret_cast<uintptr_t>(dst);
    if (s < d + (uintptr_t)bytes && d < s + (uintptr_t)bytes) return SSM_ERR_ALIAS;
    // the source must be page-locked host memory (readable by the device), the
    // destination device memory: anything else is refused before a launch
    if (!is_host_locked(src) || !is_host_locked(static_cast<const char *>(src) + (bytes - 1)) || !is_device(dst))
        return SSM_ERR_UNSUPPORTED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const long long cap = 2LL * sm_count();  // two 512-thread blocks per SM
    if (s % 16 == 0 && d % 16 == 0) {
        const long long nvec = bytes / 16;
        const int ntail = (int)(bytes % 16);
        const long long blocks = nvec > 0 ? std::min<long long>(cap, (nvec + kPullThreads - 1) / kPullThreads) : 1;
        ssm_pull_kernel<<<(unsigned)blocks, kPullThreads, 0, st>>>(
            static_cast<uint4 *>(dst), static_cast<const uint4 *>(src), nvec,
            static_cast<unsigned char *>(dst) + nvec * 16, static_cast<const unsigned char *>(src) + nvec * 16, ntail);
    } else {
        const long long blocks = std::min<long long>(cap, (bytes + kPullThreads - 1) / kPullThreads);
        ssm_pull_bytes_kernel<<<(unsigned)blocks, kPullThreads, 0, st>>>(
            static_cast<unsigned char *>(dst), static_cast<const unsigned char *>(src), bytes);
    }
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        ssm_internal::set_last_cuda_error((int)e);
        return SSM_ERR_CUDA;
    }
    return SSM_OK;
}

int ssm_copy_from_host_n(const ssm_copy_segment_t *segs, int32_t nseg, void *stream) {
    if (nseg < 0 || nseg > SSM_COPY_MAX_SEGMENTS) return SSM_ERR_SHAPE;
    if (nseg == 0) return SSM_OK;
    if (segs == nullptr) return SSM_ERR_NULL;
    // shapes, pointers and overlaps first, then what the pointers point to
    for (int i = 0; i < nseg; ++i) {
        if (segs[i].bytes < 0) return SSM_ERR_SHAPE;
        if (segs[i].bytes > 0 && (segs[i].dst == nullptr || segs[i].src == nullptr)) return SSM_ERR_NULL;
    }
    for (int i = 0; i < nseg; ++i) {
        const ssm_copy_segment_t &g = segs[i];
        if (g.bytes == 0) continue;
        const uintptr_t d = reinterpret_cast<uintptr_t>(g.dst);
        for (int k = 0; k < nseg; ++k) {  // a destination overlaps no source and no other destination
            const ssm_copy_segment_t &o = segs[k];
            if (o.bytes == 0) continue;
            const uintptr_t os = reinterpret_cast<uintptr_t>(o.src), od = reinterpret_cast<uintptr_t>(o.dst);
            if (os < d + (uintptr_t)g.bytes && d < os + (uintptr_t)o.bytes) return SSM_ERR_ALIAS;
            if (k != i && od < d + (uintptr_t)g.bytes && d < od + (uintptr_t)o.bytes) return SSM_ERR_ALIAS;
        }
    }
    bool aligned16 = true;
    int live = 0;
    for (int i = 0; i < nseg; ++i) {
        const ssm_copy_segment_t &g = segs[i];
        if (g.bytes == 0) continue;
        if (!is_host_locked(g.src) || !is_host_locked(static_cast<const char *>(g.src) + (g.bytes - 1)) ||
            !is_device(g.dst))
            return SSM_ERR_UNSUPPORTED;
        aligned16 = aligned16 && reinterpret_cast<uintptr_t>(g.src) % 16 == 0 &&
                    reinterpret_cast<uintptr_t>(g.dst) % 16 == 0;
        ++live;
    }
    if (live == 0) return SSM_OK;
    if (!aligned16) {  // each segment on its own
        for (int i = 0; i < nseg; ++i) {
            if (segs[i].bytes == 0) continue;
            const int rc = ssm_copy_from_host(segs[i].dst, segs[i].src, segs[i].bytes, stream);
            if (rc != SSM_OK) return rc;
        }
        return SSM_OK;
    }
    PullSegs sg{};
    long long run = 0;
    for (int i = 0; i < nseg; ++i) {
        if (segs[i].bytes == 0) continue;
        sg.dst[sg.n] = static_cast<uint4 *>(segs[i].dst);
        sg.src[sg.n] = static_cast<const uint4 *>(segs[i].src);
        run += segs[i].bytes / 16;
        sg.end[sg.n] = run;
        sg.tail[sg.n] = (int)(segs[i].bytes % 16);
        ++sg.n;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const long long cap = 2LL * sm_count();
    const long long blocks = run > 0 ? std::min<long long>(cap, (run + kPullThreads - 1) / kPullThreads) : 1;
    if (run == 0) {  // tails only: keep end[] increasing for the search (it is not entered)
        for (int k = 0; k < sg.n; ++k) sg.end[k] = 0;
    }
    ssm_pull_segments_kernel<<<(unsigned)blocks, kPullThreads, 0, st>>>(sg);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        ssm_internal::set_last_cuda_error((int)e);
        return SSM_ERR_CUDA;
    }
    return SSM_OK;
}

}  // extern "C"
