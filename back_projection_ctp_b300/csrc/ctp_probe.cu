// Bandwidth probes for the benchmark's L2 roofline (measurement only; not part
// of the projector library).
//
// The projector's segment stream is served by L1 and L2, not DRAM: the
// backward's float reductions travel from L1 to L2 in 32-byte sectors and the
// forward's gathers hit in L1 / L2.  The roofline that bounds them is therefore
// the rate at which L2 takes reductions (and serves loads), which these probes
// measure on the machine they run on:
//
//   ctp_probe_l2_reduction  every warp instruction is a float reduction of 32
//                           consecutive floats (4 full sectors) into a buffer
//                           that stays in L2: the highest rate at which useful
//                           reduction bytes reach L2 (8 floats per sector).
//                           sparse = 1: each lane reduces one float into its own
//                           sector instead (1 float per sector), the sector rate.
//   ctp_probe_l2_load       coalesced 16-byte loads that bypass L1 (ld.global.cg)
//                           from a buffer that stays in L2.
//   ctp_probe_smem_accumulate  float accumulation in shared memory: atomics,
//                           plain load-add-store, and atomics with 4 lanes per
//                           word (a work-layout question of the backward walks).
//   ctp_probe_l2_bulk_reduction  the async copy engine's bulk reductions of
//                           shared-memory runs into the same kind of buffer
//                           (full sectors): whether L2 takes them faster than
//                           a dense stream of float reductions.
//
// Both walk the buffer with a per-warp stride so that concurrent warps touch
// different lines; the caller times them with CUDA events on `stream`.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

__global__ void __launch_bounds__(256) probe_red_kernel(float *__restrict__ buf, long long n,
                                                        int iters, int sparse)
{
    const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    const long long span = sparse ? 256 : 32;  // floats one warp instruction covers
    const long long lines = n / span;
    long long line = warp % lines;
    const float v = 1.0f + 1e-3f * lane;
    for (int it = 0; it < iters; ++it) {
        const long long base = line * span;
        atomicAdd(buf + base + (sparse ? 8 * lane : lane), v);
        line += nwarps;
        if (line >= lines) line -= lines;
    }
}

__global__ void __launch_bounds__(256) probe_load_kernel(const float4 *__restrict__ buf,
                                                         long long n4, int iters,
                                                         float *__restrict__ sink)
{
    const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    const long long lines = n4 / 32;
    long long line = warp % lines;
    float acc = 0.0f;
    for (int it = 0; it < iters; ++it) {
        const float4 q = __ldcg(buf + line * 32 + lane);
        acc += q.x + q.y + q.z + q.w;
        line += nwarps;
        if (line >= lines) line -= lines;
    }
    if (acc == 1.2345e-30f) sink[0] = acc;  // keeps the loads; never true for the probe's data
}

// Shared-memory float accumulation: every thread adds `iters` times into its
// own word of a block-wide array (no two lanes on one word).  mode 0: atomicAdd
// on shared memory; mode 1: plain load, add and store; mode 2: atomicAdd where
// the 32 lanes of a warp share 8 words (4 lanes per word).
__global__ void __launch_bounds__(256) probe_smem_kernel(int iters, int mode, float *__restrict__ sink)
{
    __shared__ float acc[256];
    acc[threadIdx.x] = 0.0f;
    __syncthreads();
    const int w = mode == 2 ? (threadIdx.x & ~31) + ((threadIdx.x & 31) >> 2) : threadIdx.x;
    const float v = 1.0f + 1e-3f * (threadIdx.x & 31);
    if (mode == 1) {
        for (int it = 0; it < iters; ++it) {
            volatile float *a = acc;
            a[w] = a[w] + v;
        }
    } else {
        for (int it = 0; it < iters; ++it) atomicAdd(acc + w, v);
    }
    __syncthreads();
    if (acc[threadIdx.x] == 1.2345e-30f) sink[0] = acc[threadIdx.x];
}

// Bulk reductions (the async copy engine's cp.reduce.async.bulk .add.f32): the
// first `lanes` lanes of every warp each add a `bytes`-long run of shared
// memory into the next run of buf, at most 8 runs in flight per thread.
__global__ void __launch_bounds__(256) probe_bulk_red_kernel(float *__restrict__ buf, long long n,
                                                             int iters, int bytes, int lanes)
{
    __shared__ __align__(128) float src[1024];
    for (int i = threadIdx.x; i < 1024; i += blockDim.x) src[i] = 1.0f + 1e-3f * (i & 31);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    const int lane = threadIdx.x & 31;
    if (lane >= lanes) return;
    const unsigned s = (unsigned)__cvta_generic_to_shared(src);
    const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long issuers = (((long long)gridDim.x * blockDim.x) >> 5) * lanes;
    const long long seg = bytes / 4;
    const long long segs = n / seg;
    long long g = warp * lanes + lane;
    for (int it = 0; it < iters; ++it) {
        asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;"
                     :: "l"(buf + g * seg), "r"(s), "r"(bytes) : "memory");
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        asm volatile("cp.async.bulk.wait_group.read 8;" ::: "memory");
        g += issuers;
        if (g >= segs) g -= segs;
    }
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

int blocks_for(int sms) { return sms * 8; }

}  // namespace

extern "C" {

// Adds to buf[0, n): grid of 8 blocks of 256 threads per SM, `iters` reductions
// per thread; n / (32 floats, or 256 when sparse) must be at least the grid's
// warps.  Returns 0, 1 (bad arguments) or 9 (launch failed).  Useful bytes per launch:
// 4 * (threads) * iters.
int ctp_probe_l2_reduction(float *buf, long long n, int iters, int sparse, void *stream)
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 9;
    // every warp must own a distinct line: the walk wraps with one subtraction
    const long long span = sparse ? 256 : 32, warps = (long long)blocks_for(sms) * 256 / 32;
    if (!buf || n < 256 || iters < 1 || n / span < warps) return 1;
    probe_red_kernel<<<blocks_for(sms), 256, 0, (cudaStream_t)stream>>>(buf, n, iters,
                                                                        sparse ? 1 : 0);
    return cudaGetLastError() == cudaSuccess ? 0 : 9;
}

// Reads buf[0, n) (n a multiple of 128 floats, buf 16-byte aligned): 16 bytes per
// thread per iteration.  sink: one device float (written only in a case that
// does not occur).  Returns 0, 1 (bad arguments) or 9.
int ctp_probe_l2_load(const float *buf, long long n, int iters, float *sink, void *stream)
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 9;
    const long long warps = (long long)blocks_for(sms) * 256 / 32;
    if (!buf || !sink || n < 128 || n % 128 != 0 || ((uintptr_t)buf & 15) || iters < 1 ||
        n / 128 < warps)
        return 1;
    probe_load_kernel<<<blocks_for(sms), 256, 0, (cudaStream_t)stream>>>(
        reinterpret_cast<const float4 *>(buf), n / 4, iters, sink);
    return cudaGetLastError() == cudaSuccess ? 0 : 9;
}

// Shared-memory accumulation rate (see probe_smem_kernel): 8 blocks of 256
// threads per SM, `iters` adds per thread.  Returns 0, 1 or 9.
int ctp_probe_smem_accumulate(int iters, int mode, float *sink, void *stream)
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 9;
    if (!sink || iters < 1 || mode < 0 || mode > 2) return 1;
    probe_smem_kernel<<<blocks_for(sms), 256, 0, (cudaStream_t)stream>>>(iters, mode, sink);
    return cudaGetLastError() == cudaSuccess ? 0 : 9;
}

// Bulk-reduction rate (see probe_bulk_red_kernel): 8 blocks of 256 threads per
// SM, `lanes` (1..32) issuing lanes per warp, `iters` runs of `bytes` (16..4096,
// a multiple of 16) per issuing lane into buf[0, n) (16-byte aligned, n a
// multiple of bytes / 4, at least as many runs as issuing lanes).  Useful bytes
// per launch: bytes * issuing lanes * iters.  Returns 0, 1 or 9.
int ctp_probe_l2_bulk_reduction(float *buf, long long n, int iters, int bytes, int lanes,
                                void *stream)
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 9;
    if (!buf || ((uintptr_t)buf & 15) || iters < 1 || bytes < 16 || bytes > 4096 ||
        bytes % 16 != 0 || lanes < 1 || lanes > 32)
        return 1;
    const long long seg = bytes / 4, issuers = (long long)blocks_for(sms) * 256 / 32 * lanes;
    if (n % seg != 0 || n / seg < issuers) return 1;
    probe_bulk_red_kernel<<<blocks_for(sms), 256, 0, (cudaStream_t)stream>>>(buf, n, iters, bytes,
                                                                             lanes);
    return cudaGetLastError() == cudaSuccess ? 0 : 9;
}

// SM count of the current device (the probes' grid is 8 blocks of 256 threads per SM).
int ctp_probe_sm_count(int *out)
{
    int dev = 0;
    if (!out || cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 9;
    return 0;
}

}  // extern "C"
