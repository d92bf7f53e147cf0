/*
 * synth_dev.cu - device side of the seeded input generator (see synth.h).
 * Fills device buffers with exactly the bits synth_host.c produces, so that
 * full-size workloads (tens of GB of bf16 weights) are made in milliseconds
 * on the GPU while the oracle regenerates any rows it samples on the host.
 */
#include <cuda_runtime.h>
#include <stdint.h>

#include "synth.h"

namespace {

__global__ void k_weights(uint64_t key, uint64_t kc, uint64_t kg, int64_t N, int64_t K, int outliers,
                          uint16_t* out) {
  int64_t n = blockIdx.y + (int64_t)blockIdx.z * gridDim.y;
  if (n >= N) return;
  float scale = syn_channel_scale(key, (uint64_t)n);
  for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < K; k += (int64_t)gridDim.x * blockDim.x)
    out[n * K + k] = syn_weight_ex(kc, kg, (uint64_t)n * (uint64_t)K + (uint64_t)k, scale, outliers);
}

__global__ void k_activations(uint64_t key, int64_t count, uint16_t* out) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += (int64_t)gridDim.x * blockDim.x)
    out[i] = syn_activation(key, (uint64_t)i);
}

}  // namespace

extern "C" {

/* N x K bf16 weight matrix (seed, layer, tensor) into device memory out[N*K]; outliers = 0 gives
 * the head recipe. Returns a cudaError_t. */
int syn_weights_dev_ex(uint64_t seed, uint64_t layer, uint64_t tensor, int64_t N, int64_t K, int outliers, void* out,
                       void* stream) {
  if (N <= 0 || K <= 0) return 0;
  uint64_t key = syn_key(seed, layer, tensor);
  int64_t gy = N < 65535 ? N : 65535;
  int64_t gz = (N + gy - 1) / gy;
  int gx = (int)((K + 255) / 256);
  if (gx > 64) gx = 64;
  dim3 grid((unsigned)gx, (unsigned)gy, (unsigned)gz);
  k_weights<<<grid, 256, 0, (cudaStream_t)stream>>>(key, syn_substream(key, SYN_S_CAT), syn_substream(key, SYN_S_GAUSS),
                                                    N, K, outliers, (uint16_t*)out);
  return (int)cudaGetLastError();
}

int syn_weights_dev(uint64_t seed, uint64_t layer, uint64_t tensor, int64_t N, int64_t K, void* out, void* stream) {
  return syn_weights_dev_ex(seed, layer, tensor, N, K, 1, out, stream);
}

/* count bf16 N(0,1) activations (seed, layer, tensor) into device memory. */
int syn_activations_dev(uint64_t seed, uint64_t layer, uint64_t tensor, int64_t count, void* out, void* stream) {
  if (count <= 0) return 0;
  int64_t blocks = (count + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  k_activations<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(syn_key(seed, layer, tensor), count, (uint16_t*)out);
  return (int)cudaGetLastError();
}

}  // extern "C"
