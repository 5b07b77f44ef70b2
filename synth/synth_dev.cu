// synth_dev.cu -- device fill kernels for the counter-based input generator.
// Same definitions as synth.c (stated in synth.h): integer streams and the
// fp16 scale stream only (the Box-Muller normals are drawn on the host).
// Used to put multi-GB synthetic expert weights into HBM quickly; a GPU test
// checks these bytes against the host generator.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define SYNTH_GOLDEN 0x9E3779B97F4A7C15ull

__device__ __forceinline__ uint64_t mix64_dev(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static uint64_t mix64_host(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__global__ void fill_int8_kernel(int8_t *out, uint64_t n, uint64_t key, uint64_t first) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t j = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += stride) {
    uint64_t r = mix64_dev(key + (first + j + 1) * SYNTH_GOLDEN);
    out[j] = (int8_t)(-127 + (int)(((r >> 40) * 255u) >> 24));
  }
}

__global__ void fill_code2_kernel(uint8_t *out, uint64_t n, uint64_t key, uint64_t first) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t j = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += stride) {
    uint64_t r = mix64_dev(key + (first + j + 1) * SYNTH_GOLDEN);
    out[j] = (uint8_t)(r >> 56);
  }
}

__global__ void fill_scale_kernel(__half *out, uint64_t n, uint64_t key, uint64_t first,
                                  double denom) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t j = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += stride) {
    uint64_t r = mix64_dev(key + (first + j + 1) * SYNTH_GOLDEN);
    double u = (double)(r >> 11) * 0x1.0p-53;
    out[j] = __double2half(__ddiv_rn(__dadd_rn(0.5, u), denom));
  }
}

static int grid_for(uint64_t n) {
  uint64_t g = (n + 255) / 256;
  if (g > 152ull * 64) g = 152ull * 64;
  if (g < 1) g = 1;
  return (int)g;
}

static uint64_t key_of(uint64_t seed, uint64_t stream) {
  return mix64_host((seed << 32) | (stream & 0xFFFFFFFFull));
}

extern "C" int synth_dev_int8(void *out, uint64_t seed, uint64_t stream, uint64_t first,
                              uint64_t n, void *stream_handle) {
  if (n == 0) return 0;
  fill_int8_kernel<<<grid_for(n), 256, 0, (cudaStream_t)stream_handle>>>(
      (int8_t *)out, n, key_of(seed, stream), first);
  return (int)cudaGetLastError();
}

extern "C" int synth_dev_code2(void *out, uint64_t seed, uint64_t stream, uint64_t first,
                               uint64_t n, void *stream_handle) {
  if (n == 0) return 0;
  fill_code2_kernel<<<grid_for(n), 256, 0, (cudaStream_t)stream_handle>>>(
      (uint8_t *)out, n, key_of(seed, stream), first);
  return (int)cudaGetLastError();
}

extern "C" int synth_dev_scale_f16(void *out, uint64_t seed, uint64_t stream, uint64_t first,
                                   uint64_t n, double denom, void *stream_handle) {
  if (n == 0) return 0;
  fill_scale_kernel<<<grid_for(n), 256, 0, (cudaStream_t)stream_handle>>>(
      (__half *)out, n, key_of(seed, stream), first, denom);
  return (int)cudaGetLastError();
}
