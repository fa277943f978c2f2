// Seeded synthetic inputs for the rotated 4-bit KV-cache decode path.
//
// This module only draws numbers. It holds none of the method's arithmetic: no
// normalisation, rotation, quantisation or attention. Both the CUDA path (bench
// and GPU tests fill caches with it) and the CPU oracle's tests take their inputs
// from here, so the two sides see the same bits.
//
// Generator: splitmix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
// generators", OOPSLA 2014), used counter-style: draw(key, n) is the (n+1)-th
// output of a splitmix64 stream whose state starts at `key`, so any element can
// be regenerated on its own.
//
// Normals: Irwin-Hall with twelve 16-bit uniforms, summed as integers. The sum is
// converted once and scaled by 2^-16, which is exact in fp32, so host and device
// produce identical floats. Support is [-6, 6], variance 1.
//
// Host functions are multithreaded with std::thread; device functions launch one
// elementwise kernel on the caller's stream.

#include <cuda_runtime.h>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>
#include <algorithm>

#define SYN_HD __host__ __device__ __forceinline__

namespace {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;

SYN_HD uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

SYN_HD uint64_t draw(uint64_t key, uint64_t n) { return mix64(key + kGolden * (n + 1)); }

SYN_HD float normal_at(uint64_t key, uint64_t i) {
  int32_t s = 0;
#pragma unroll
  for (int w = 0; w < 3; ++w) {
    uint64_t u = draw(key, 3 * i + w);
    s += (int32_t)(u & 0xFFFF) + (int32_t)((u >> 16) & 0xFFFF) + (int32_t)((u >> 32) & 0xFFFF) +
         (int32_t)(u >> 48);
  }
  // sum of twelve (u_k + 1/2)/65536 minus 6  ==  (s + 6 - 6*65536) / 65536
  return (float)(s - 393210) * (1.0f / 65536.0f);
}

SYN_HD float uniform_at(uint64_t key, uint64_t i) {
  return (float)(draw(key, i) >> 40) * (1.0f / 16777216.0f);
}

SYN_HD uint16_t bf16_rne_bits(float x) {
  uint32_t u;
#ifdef __CUDA_ARCH__
  u = __float_as_uint(x);
#else
  std::memcpy(&u, &x, 4);
#endif
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x40);  // quiet NaN
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

struct Mult128 {
  float m[128];
};

// dtype: 0 = fp32 output, 1 = bf16 output (round to nearest even)
__global__ void normal_fill_kernel(uint64_t key, uint64_t start, int64_t n, Mult128 mult, int use_mult,
                                   int dtype, void* out) {
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (int64_t)gridDim.x * blockDim.x) {
    uint64_t i = start + (uint64_t)e;
    float x = normal_at(key, i);
    if (use_mult) x = __fmul_rn(x, mult.m[i & 127]);
    if (dtype == 0)
      static_cast<float*>(out)[e] = x;
    else
      static_cast<uint16_t*>(out)[e] = bf16_rne_bits(x);
  }
}

template <class F>
void parallel_for(int64_t n, F f) {
  int nt = (int)std::max(1u, std::thread::hardware_concurrency());
  if (n < (int64_t)1 << 16) nt = 1;
  nt = (int)std::min<int64_t>(nt, 64);
  std::vector<std::thread> th;
  int64_t per = (n + nt - 1) / nt;
  for (int t = 0; t < nt; ++t) {
    int64_t a = t * per, b = std::min(n, a + per);
    if (a >= b) break;
    th.emplace_back([=] { f(a, b); });
  }
  for (auto& x : th) x.join();
}

}  // namespace

extern "C" {

uint64_t synth_key(uint64_t seed, uint64_t stream) { return mix64(seed + kGolden * (stream + 1)); }

uint64_t synth_draw(uint64_t key, uint64_t n) { return draw(key, n); }

// out[e] = normal(start + e) * mult[(start + e) % 128]   (mult may be null)
void synth_normal_host(uint64_t key, uint64_t start, int64_t n, const float* mult, int dtype, void* out) {
  parallel_for(n, [&](int64_t a, int64_t b) {
    for (int64_t e = a; e < b; ++e) {
      uint64_t i = start + (uint64_t)e;
      float x = normal_at(key, i);
      if (mult) x = x * mult[i & 127];
      if (dtype == 0)
        static_cast<float*>(out)[e] = x;
      else
        static_cast<uint16_t*>(out)[e] = bf16_rne_bits(x);
    }
  });
}

void synth_uniform_host(uint64_t key, uint64_t start, int64_t n, float* out) {
  parallel_for(n, [&](int64_t a, int64_t b) {
    for (int64_t e = a; e < b; ++e) out[e] = uniform_at(key, start + (uint64_t)e);
  });
}

// Raw 64-bit draws (used for integer choices: lengths, permutations, channel picks).
void synth_draw_host(uint64_t key, uint64_t start, int64_t n, uint64_t* out) {
  for (int64_t e = 0; e < n; ++e) out[e] = draw(key, start + (uint64_t)e);
}

// Fisher-Yates permutation of 0..n-1 driven by draw(key, i).
void synth_permutation_host(uint64_t key, int64_t n, int32_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)i;
  for (int64_t i = n - 1; i > 0; --i) {
    int64_t j = (int64_t)(draw(key, (uint64_t)i) % (uint64_t)(i + 1));
    std::swap(out[i], out[j]);
  }
}

// Device fill with the same definition. Returns 0 or a cudaError_t value.
int synth_normal_device(uint64_t key, uint64_t start, int64_t n, const float* mult_host, int dtype,
                        void* out_dev, void* stream) {
  if (n <= 0) return 0;
  Mult128 m;
  int use = mult_host != nullptr;
  for (int i = 0; i < 128; ++i) m.m[i] = use ? mult_host[i] : 1.0f;
  int64_t blocks = std::min<int64_t>((n + 255) / 256, 152 * 16);
  normal_fill_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(key, start, n, m, use, dtype,
                                                                           out_dev);
  return (int)cudaGetLastError();
}

}  // extern "C"
