// A wait that can never finish, run through the bounded mbarrier wait every
// libpa kernel uses (mbar_wait in pa_device.cuh): it must give up within
// about a second, report PA_DEVERR_TIMEOUT in the device error word and
// leave the context usable (a second kernel then waits on a barrier that
// was arrived at and finishes at once).  One thread, one barrier in shared
// memory; nothing is read or written outside the two result buffers.
// Prints one JSON line; exit status 0 when every check holds.
#include <cstdio>

#include <cuda_runtime.h>

#include "pa_device.cuh"

namespace {

__global__ void wait_on_unarrived_barrier(int *done, unsigned long long *elapsed_ns) {
    __shared__ __align__(8) uint64_t bar;
    pa::mbar_init(&bar, 1);          // one arrival expected; none ever comes
    pa::fence_mbar_init();
    const uint64_t t0 = pa::global_ns();
    const bool ok = pa::mbar_wait(&bar, 0);
    const uint64_t t1 = pa::global_ns();
    done[0] = ok ? 1 : 0;
    elapsed_ns[0] = t1 - t0;
}

__global__ void wait_after_arrival(int *done) {
    __shared__ __align__(8) uint64_t bar;
    pa::mbar_init(&bar, 1);
    pa::fence_mbar_init();
    pa::mbar_arrive(&bar);           // the phase completes
    done[0] = pa::mbar_wait(&bar, 0) ? 1 : 0;
}

}  // namespace

int main() {
    int *d_done = nullptr;
    unsigned long long *d_ns = nullptr;
    if (cudaMalloc(&d_done, sizeof(int)) != cudaSuccess || cudaMalloc(&d_ns, sizeof(unsigned long long)) != cudaSuccess) {
        std::printf("{\"error\": \"cudaMalloc failed\"}\n");
        return 2;
    }
    const int unset = -1;
    cudaMemcpy(d_done, &unset, sizeof(int), cudaMemcpyHostToDevice);
    wait_on_unarrived_barrier<<<1, 1>>>(d_done, d_ns);
    const cudaError_t e1 = cudaDeviceSynchronize();
    int done1 = -1, word = 0;
    unsigned long long ns = 0;
    cudaMemcpy(&done1, d_done, sizeof(int), cudaMemcpyDeviceToHost);
    cudaMemcpy(&ns, d_ns, sizeof(ns), cudaMemcpyDeviceToHost);
    cudaMemcpyFromSymbol(&word, pa::g_device_error, sizeof(int));

    cudaMemcpy(d_done, &unset, sizeof(int), cudaMemcpyHostToDevice);
    wait_after_arrival<<<1, 1>>>(d_done);
    const cudaError_t e2 = cudaDeviceSynchronize();
    int done2 = -1;
    cudaMemcpy(&done2, d_done, sizeof(int), cudaMemcpyDeviceToHost);

    const double ms = ns / 1e6;
    std::printf("{\"first\": \"%s\", \"first_wait_completed\": %d, \"first_wait_ms\": %.1f, \"error_word\": %d, "
                "\"second\": \"%s\", \"second_wait_completed\": %d}\n",
                cudaGetErrorString(e1), done1, ms, word, cudaGetErrorString(e2), done2);
    const bool pass = e1 == cudaSuccess && done1 == 0 && (word & PA_DEVERR_TIMEOUT) && ms > 10.0 && ms < 5000.0 &&
                      e2 == cudaSuccess && done2 == 1;
    cudaFree(d_done);
    cudaFree(d_ns);
    return pass ? 0 : 1;
}
