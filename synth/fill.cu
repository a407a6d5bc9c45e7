// fill.cu -- device twin of synth.expert_record(): writes seeded MXFP4 expert records
// straight into device memory.  Input generation only (no arithmetic of the MoE layer).
//
// SplitMix64 (Steele, Lea & Flood, OOPSLA 2014): output i of the stream keyed by k is
// mix(k + (i + 1) * 0x9E3779B97F4A7C15), mix the SplitMix64 finaliser.  Operand keys:
//   k = mix(mix(mix(seed + G) + layer) + expert * 8 + op),  G = 0x9E3779B97F4A7C15.
// Packed operands: byte b is byte (b % 8) (little endian) of output b / 8.
// Scale operands: byte b = lo + ((output_b >> 32) * (hi - lo + 1) >> 32).
#include <cstdint>
#include <cuda_runtime.h>

namespace {
constexpr uint64_t kG = 0x9E3779B97F4A7C15ull;
__device__ __forceinline__ uint64_t mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}
__device__ __forceinline__ uint64_t out(uint64_t key, uint64_t i) { return mix(key + (i + 1) * kG); }

struct Layout { long long off[7]; };

__global__ void k_fill(uint8_t *base, long long stride, int e0, int ne, unsigned long long seed,
                       int layer, Layout L, int lo, int hi) {
  const long long words = L.off[6] / 8;
  const long long n = (long long)ne * words;
  const uint64_t span = (uint64_t)(hi - lo + 1);
  const uint64_t k0 = mix(mix(seed + kG) + (uint64_t)layer);
  for (long long q = blockIdx.x * (long long)blockDim.x + threadIdx.x; q < n;
       q += (long long)gridDim.x * blockDim.x) {
    const int e = e0 + (int)(q / words);
    const long long b = (q % words) * 8;
    int op = 0;
    while (op < 5 && b >= L.off[op + 1]) op++;
    const uint64_t key = mix(k0 + (uint64_t)e * 8 + (uint64_t)op);
    const long long rel = b - L.off[op];
    uint64_t v;
    if (op == 0 || op == 2 || op == 4) {
      v = out(key, (uint64_t)(rel / 8));
    } else {
      v = 0;
      for (int k = 0; k < 8; k++) {
        const uint64_t h = out(key, (uint64_t)(rel + k)) >> 32;
        const uint64_t s = (uint64_t)lo + ((h * span) >> 32);
        v |= (s & 0xffull) << (8 * k);
      }
    }
    *reinterpret_cast<uint64_t *>(base + (long long)(e - e0) * stride + b) = v;
  }
}
}  // namespace

// Fill experts [e0, e0 + ne) of one layer at base (expert e0 at base), records of the
// given operand offsets (off[6] = record size, a multiple of 16), stride bytes apart.
extern "C" int k3synth_fill_experts(void *base, long long stride, int e0, int ne,
                                    unsigned long long seed, int layer, const long long *off,
                                    int scale_lo, int scale_hi, void *stream) {
  if (!base || !off || ne < 0 || stride % 16 || off[6] % 16 || stride < off[6]) return 1;
  if (ne == 0) return 0;
  Layout L;
  for (int i = 0; i < 7; i++) L.off[i] = off[i];
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  k_fill<<<sms * 8, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<uint8_t *>(base), stride, e0, ne, seed, layer, L, scale_lo, scale_hi);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}
