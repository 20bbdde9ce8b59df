// zero1_checksum.cu - exact, order-independent checksum of a buffer: the
// silent-data-corruption guard for the replicated parameters.

#include "zero1_device.cuh"
#include "zero1_checks.h"

namespace {

// ----------------------------------------------- consistency checksum -----
//
// Silent-data-corruption guard for the replicated parameters ("CS336 Lecture
// 7: Parallelism 1" case studies): over a buffer's 16-bit units u_i,
// out[0] = sum u_i and out[1] = sum (i + 1) u_i, both mod 2^64.  Integer sums
// are exact, so the per-thread partial sums, the warp reduction and the
// atomicAdd of each warp's partials give the same words in any order.

__device__ __forceinline__ void warp_sum_u64(uint64_t &x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
}

// Units j and j + 1 packed in one 32-bit word (j in the low half).
__device__ __forceinline__ void add_pair(uint32_t word, int64_t j, uint64_t &s1, uint64_t &s2)
{
    const uint64_t lo = word & 0xffffu, hi = word >> 16;
    s1 += lo + hi;
    s2 += (uint64_t)(j + 1) * lo + (uint64_t)(j + 2) * hi;
}

__global__ void __launch_bounds__(kBlock)
k_checksum16(const uint16_t *__restrict__ u, const Walk w, unsigned long long *out)
{
    const int64_t tid = grid_tid();
    const int64_t nthr = grid_threads();
    uint64_t s1 = 0, s2 = 0;
    for (int64_t i = tid; i < w.nvec; i += nthr) {
        const int64_t j = w.head + i * kVec;
        const uint4 q = ld_stream_u4(u + j);
        add_pair(q.x, j, s1, s2);
        add_pair(q.y, j + 2, s1, s2);
        add_pair(q.z, j + 4, s1, s2);
        add_pair(q.w, j + 6, s1, s2);
    }
    const int64_t ns = w.L - w.nvec * kVec;
    for (int64_t q = tid; q < ns; q += nthr) {
        const int64_t j = scalar_index(w, q);
        const uint64_t x = ld_stream_u16(u + j);
        s1 += x;
        s2 += (uint64_t)(j + 1) * x;
    }
    warp_sum_u64(s1);
    warp_sum_u64(s2);
    if ((threadIdx.x & 31) == 0 && (s1 | s2)) {
        atomicAdd(out, (unsigned long long)s1);
        atomicAdd(out + 1, (unsigned long long)s2);
    }
}

}  // namespace

extern "C" int zero1_checksum(const void *data, int64_t nbytes, uint64_t *out, zero1_stream_t stream)
{
    Z1Trace trace("zero1_checksum");
    if (!out) return z1_fail(ZERO1_EINVAL, "checksum: out is NULL");
    if (((uintptr_t)out & 7u) != 0) return z1_fail(ZERO1_EALIGN, "checksum: out is not 8-byte aligned");
    if (nbytes < 0 || (nbytes & 1)) return z1_fail(ZERO1_EINVAL, "checksum: %lld bytes is not a whole number of "
                                                   "16-bit units", (long long)nbytes);
    if (nbytes > 0 && !data) return z1_fail(ZERO1_EINVAL, "checksum: data is NULL");
    int rc;
    if ((rc = check_natural(data, 2, "checksum data")) != ZERO1_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(out, 0, 2 * sizeof(uint64_t), st);
    if (e != cudaSuccess) return z1_fail(ZERO1_ECUDA, "checksum: clearing out: %s", cudaGetErrorString(e));
    const int64_t U = nbytes / 2;
    if (U == 0) return ZERO1_OK;
    const ArrayRef arr[1] = {{data, 2}};
    const Walk w = make_walk(U, U, arr, 1);
    const int grid = grid_for(k_checksum16, w);
    k_checksum16<<<grid, kBlock, 0, st>>>(static_cast<const uint16_t *>(data), w,
                                         reinterpret_cast<unsigned long long *>(out));
    return launch_status("checksum launch");
}
