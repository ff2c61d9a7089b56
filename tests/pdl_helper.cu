// pdl_helper.cu -- test-only kernel for the ordering tests of the decode calls.
//
// delayed_copy lets the next kernel of the stream start at once (it triggers
// its dependents on entry, as a producer kernel under programmatic launch may),
// then waits `delay_ns` of %globaltimer and only then copies n int32 values.  A
// consumer launched right after it that read those values before its
// programmatic wait would see the old ones.  The wait is bounded by time and by
// an iteration count, so it always ends.
#include <cuda_runtime.h>
#include <stdint.h>

__global__ void delayed_copy_kernel(int32_t* dst, const int32_t* src, int n,
                                    unsigned long long delay_ns) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    unsigned long long t0, t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    for (int i = 0; i < (1 << 24); ++i) {
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        if (t - t0 >= delay_ns) break;
    }
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
        dst[i] = src[i];
}

extern "C" int pdl_delayed_copy(int32_t* dst, const int32_t* src, int n,
                                unsigned long long delay_ns, void* stream) {
    delayed_copy_kernel<<<1, 128, 0, static_cast<cudaStream_t>(stream)>>>(dst, src, n, delay_ns);
    return static_cast<int>(cudaGetLastError());
}
