// Test helper: raw Philox4x32-10 words from cuRAND's device API, to pin the oracle's
// generator (its constants, rounds and counter/key layout) against a library
// implementation.  curand_init(seed, subsequence, offset) with offset = 4q and
// subsequence = stream positions the generator at counter (q, stream) under key
// (seed low, seed high); curand4 then returns that block's four words.
#include <cstdint>
#include <cuda_runtime.h>
#include <curand_kernel.h>

__global__ void words_kernel(unsigned long long seed, unsigned long long stream, unsigned long long q0,
                             int nblocks, uint4* out) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= nblocks) return;
  curandStatePhilox4_32_10_t st;
  curand_init(seed, stream, 4ull * (q0 + (unsigned long long)b), &st);
  out[b] = curand4(&st);
}

// Fills host `out` with nblocks x 4 words for counters q0 .. q0+nblocks-1.  Returns 0 on
// success, else the CUDA error code.
extern "C" int curand_philox_words(unsigned long long seed, unsigned long long stream, unsigned long long q0,
                                   int nblocks, unsigned int* out) {
  uint4* d = nullptr;
  cudaError_t e = cudaMalloc(&d, sizeof(uint4) * (size_t)nblocks);
  if (e != cudaSuccess) return (int)e;
  words_kernel<<<(nblocks + 127) / 128, 128>>>(seed, stream, q0, nblocks, d);
  e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaMemcpy(out, d, sizeof(uint4) * (size_t)nblocks, cudaMemcpyDeviceToHost);
  cudaFree(d);
  return (int)e;
}
