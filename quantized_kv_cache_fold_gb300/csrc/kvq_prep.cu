// Append-time kernels of the rotated 4-bit KV cache and of the FP8 sliding-window cache.
//
// prep_kernel: "Serving Kolibri-1 with a 4-bit KV cache", section "What we do". One warp
// per key/value token-head: RMS norm and the fixed 128x128 matrix M_k = R on the key
// (the fused Q/K prologue), then 4-bit codes with an fp16 scale and offset for the key
// and for the unrotated value, written into the page slot. The same kernel applies the
// query prologue q~ = M_q n(q) (M_q = R diag(g_q g_k)) for the attention that follows.
// Blocks with blockIdx.x < kv_blocks do key/value work with M_k in shared memory; the
// rest do query rows with M_q.
//
// Every floating-point step uses explicit IEEE round-to-nearest intrinsics in the order
// fixed by the specification in kvq.h, so the codes are bit-identical to a plain CPU
// evaluation of the same formula. Two prologue specifications: the 128x128 matrix product
// (kvq_fold_qk) and the fast Walsh-Hadamard form (kvq_fold_qk_fwht), selected per call.

#include <algorithm>

#include <mutex>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kPrepWarps = 8;
constexpr int kPrepThreads = kPrepWarps * 32;
constexpr int kMStride = 129;  // padded row stride of the matrix in shared memory (conflict-free)
constexpr int kPrepSmem = (128 * kMStride + kPrepWarps * 128) * 4;

struct PrepParams {
  PrepJobs j;
  int kv_blocks;
  int kv_jobs;
  int q_jobs;
};

// 1 / sqrt(mean(x^2) + eps) of the 128-vector spread over the warp (lane l holds
// x[4l..4l+3]), in the specified order: per-lane fma chain, xor butterfly 16..1.
__device__ __forceinline__ float norm_inv(const float (&x)[4], float eps) {
  float t = __fmul_rn(x[0], x[0]);
  t = __fmaf_rn(x[1], x[1], t);
  t = __fmaf_rn(x[2], x[2], t);
  t = __fmaf_rn(x[3], x[3], t);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) t = __fadd_rn(t, __shfl_xor_sync(0xffffffffu, t, o));
  return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(t, 128.0f), eps)));
}

// Second specification (FWHT prologue): y = c FWHT(w n(x)), c = fp32(1/sqrt(128)), butterflies
// (u_i, u_i+h) -> (u_i + u_i+h, u_i - u_i+h) for h = 1, 2, ..., 64. Since R = H diag(s)/sqrt(128)
// this is R n(x) for w = s and R diag(g_q g_k) n(x) for w = fp32(s g_q g_k). Lane l holds
// elements 4l..4l+3 of x, w and y: h = 1, 2 inside the lane, h = 4..64 across lanes l ^ h/4.
__device__ __forceinline__ void prologue_fwht(const float4 w, const float (&x)[4], float eps, int lane,
                                              float (&y)[4]) {
  const float inv = norm_inv(x, eps);
  const float u0 = __fmul_rn(w.x, __fmul_rn(x[0], inv)), u1 = __fmul_rn(w.y, __fmul_rn(x[1], inv));
  const float u2 = __fmul_rn(w.z, __fmul_rn(x[2], inv)), u3 = __fmul_rn(w.w, __fmul_rn(x[3], inv));
  const float a0 = __fadd_rn(u0, u1), a1 = __fsub_rn(u0, u1), a2 = __fadd_rn(u2, u3), a3 = __fsub_rn(u2, u3);
  float v[4] = {__fadd_rn(a0, a2), __fadd_rn(a1, a3), __fsub_rn(a0, a2), __fsub_rn(a1, a3)};
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const bool upper = (lane & o) != 0;  // holds u_(i+h); the partner holds u_i
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float pv = __shfl_xor_sync(0xffffffffu, v[e], o);
      v[e] = upper ? __fsub_rn(pv, v[e]) : __fadd_rn(v[e], pv);
    }
  }
  const float c = __uint_as_float(0x3DB504F3u);  // fp32(1/sqrt(128))
#pragma unroll
  for (int e = 0; e < 4; ++e) y[e] = __fmul_rn(c, v[e]);
}

// y = M n(x). Lane l holds x[4l..4l+3] and returns y[l + 32u], u = 0..3.
// Ms: shared [128][kMStride] (Ms[j*kMStride + i] = M[j][i]); nbuf: shared float[128] of this warp.
__device__ __forceinline__ void prologue(const float* __restrict__ Ms, float* nbuf, const float (&x)[4], float eps,
                                         int lane, float (&y)[4]) {
  const float inv = norm_inv(x, eps);
  reinterpret_cast<float4*>(nbuf)[lane] =
      make_float4(__fmul_rn(x[0], inv), __fmul_rn(x[1], inv), __fmul_rn(x[2], inv), __fmul_rn(x[3], inv));
  __syncwarp();
  float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
  const float* m0 = Ms + lane * kMStride;
#pragma unroll 2
  for (int i = 0; i < kD; i += 4) {
    const float4 n4 = reinterpret_cast<const float4*>(nbuf)[i >> 2];
    const float nv[4] = {n4.x, n4.y, n4.z, n4.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      a0 = __fmaf_rn(m0[i + u], nv[u], a0);
      a1 = __fmaf_rn(m0[32 * kMStride + i + u], nv[u], a1);
      a2 = __fmaf_rn(m0[64 * kMStride + i + u], nv[u], a2);
      a3 = __fmaf_rn(m0[96 * kMStride + i + u], nv[u], a3);
    }
  }
  __syncwarp();
  y[0] = a0;
  y[1] = a1;
  y[2] = a2;
  y[3] = a3;
}

struct Quant4 {
  uint32_t c[4];  // codes of this lane's four elements
  uint32_t meta;  // fp16 scale | fp16 offset << 16
  int flags;
};

// int4 quantiser of one 128-vector spread over the warp (4 elements per lane).
__device__ __forceinline__ Quant4 quantize(const float (&y)[4]) {
  float mn = fminf(fminf(y[0], y[1]), fminf(y[2], y[3]));
  float mx = fmaxf(fmaxf(y[0], y[1]), fmaxf(y[2], y[3]));
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  Quant4 r;
  r.flags = 0;
  unsigned short ob = __half_as_ushort(__float2half_rd(mn));
  if ((ob & 0x7FFFu) == 0x7C00u) {  // below -65504: saturate
    ob = 0xFBFFu;
    r.flags |= KVQ_DEVERR_RANGE;
  }
  if (ob == 0x8000u) ob = 0;  // canonical +0
  const float o = __half2float(__ushort_as_half(ob));
  const float span = __fdiv_rn(__fsub_rn(mx, o), 15.0f);
  unsigned short sb = __half_as_ushort(__float2half_ru(span));
  if (sb == 0x7C00u) {
    sb = 0x7BFFu;
    r.flags |= KVQ_DEVERR_RANGE;
  }
  if (sb == 0x8000u) sb = 0;  // canonical +0 (zeros whose maximum came out as -0)
  const float s = __half2float(__ushort_as_half(sb));
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    int c = 0;
    if (s != 0.0f) c = __float2int_rn(__fdiv_rn(__fsub_rn(y[u], o), s));
    r.c[u] = (uint32_t)min(max(c, 0), 15);
  }
  r.meta = (uint32_t)sb | ((uint32_t)ob << 16);
  return r;
}

__global__ void __launch_bounds__(kPrepThreads) prep_kernel(const PrepParams p) {
  extern __shared__ __align__(16) float smem_f[];
  float* Ms = smem_f;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* nbuf = smem_f + 128 * kMStride + warp * 128;
  const PrepJobs& j = p.j;
  const bool kv_role = (int)blockIdx.x < p.kv_blocks;
  const float* M = kv_role ? j.Mk : j.Mq;
  // May overlap the previous grid on the stream. Before the wait: L2 prefetches of this warp's
  // first rows, and the folded weights (M, or the FWHT multipliers), which are complete before
  // the call (kvq.h) and are staged into shared memory now.
  const size_t rbytes = (size_t)kD * ((kv_role ? j.kv_bf16 : j.q_bf16) ? 2 : 4);
  const int job0 = kv_role ? (int)blockIdx.x * kPrepWarps + warp
                           : ((int)blockIdx.x - p.kv_blocks) * kPrepWarps + warp;
  const bool has_job0 = job0 < (kv_role ? p.kv_jobs : p.q_jobs);
  const uint8_t* r0a = nullptr;  // first job's rows (key and value, or query)
  const uint8_t* r0b = nullptr;
  if (has_job0) {
    if (kv_role) {
      r0a = static_cast<const uint8_t*>(j.k) + (size_t)job0 * rbytes;  // row index = token * Hkv + head = job
      r0b = static_cast<const uint8_t*>(j.v) + (size_t)job0 * rbytes;
    } else {
      r0a = static_cast<const uint8_t*>(j.q) + (size_t)job0 * rbytes;
    }
  }
  if (lane == 0 && r0a) prefetch_l2_bulk(r0a, (uint32_t)rbytes);
  if (lane == 0 && r0b) prefetch_l2_bulk(r0b, (uint32_t)rbytes);
  // the FWHT prologue needs only this lane's four multipliers; the matrix prologue stages M
  const float4 w4 = j.fwht ? reinterpret_cast<const float4*>(M)[lane] : make_float4(0.f, 0.f, 0.f, 0.f);
  if (!j.fwht) {
    // 16 independent 16-byte loads per thread, then the padded (conflict-free) shared stores
    constexpr int kPer = kD * kD / 4 / kPrepThreads;
    float4 v[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) v[u] = reinterpret_cast<const float4*>(M)[threadIdx.x + u * kPrepThreads];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int e = 4 * (threadIdx.x + u * kPrepThreads);
      float* d = Ms + (e >> 7) * kMStride + (e & 127);
      d[0] = v[u].x;
      d[1] = v[u].y;
      d[2] = v[u].z;
      d[3] = v[u].w;
    }
  }
  __syncthreads();
  griddep_wait();
  griddep_launch_dependents();

  const int Hkv = j.cache.num_kv_heads;
  if (kv_role) {
    for (int job = blockIdx.x * kPrepWarps + warp; job < p.kv_jobs; job += p.kv_blocks * kPrepWarps) {
      const int tok = job / Hkv, h = job - (job / Hkv) * Hkv;
      int seq, pos;
      if (j.seq_ids) {
        seq = j.seq_ids[tok];
        pos = j.positions[tok];
      } else {
        seq = tok / j.S;
        pos = j.ctx_len[seq] + (tok - seq * j.S);
      }
      if (seq < 0 || seq >= j.cache.num_seqs || pos < 0 || pos >= j.cache.max_pages_per_seq * kPage) {
        if (lane == 0) set_err(j.dev_err, KVQ_DEVERR_POS);
        continue;
      }
      const int page = j.cache.block_table[(size_t)seq * j.cache.max_pages_per_seq + pos / kPage];
      if (page < 0 || page >= j.cache.num_pages) {
        if (lane == 0) set_err(j.dev_err, KVQ_DEVERR_PAGE);
        continue;
      }
      const int slot = pos & (kPage - 1);
      uint8_t* blk = j.cache.pages + ((size_t)page * Hkv + h) * KVQ_INT4_BLOCK_BYTES;
      uint32_t* meta = reinterpret_cast<uint32_t*>(blk + 2 * kPage * kRec4);
      const size_t row = (size_t)tok * Hkv + h;

      float x[4], xv[4];  // key and value rows, loaded together
      load_row4(j.k, j.kv_bf16, row, lane, x);
      load_row4(j.v, j.kv_bf16, row, lane, xv);
      if (!warp_all_finite(x)) {
        if (lane == 0) set_err(j.dev_err, KVQ_DEVERR_NONFINITE);
      } else {
        float y[4];
        uint8_t* dst = blk + slot * kRec4;
        Quant4 q;
        if (j.fwht) {
          prologue_fwht(w4, x, j.eps, lane, y);  // lane holds y[4 lane + e]: codes 4l..4l+3 = bytes 2l, 2l+1
          q = quantize(y);
          *reinterpret_cast<uint16_t*>(dst + 16 * ((lane >> 3) ^ k_chunk_swz(slot)) + ((2 * lane) & 15)) =
              (uint16_t)((q.c[0] | (q.c[1] << 4)) | ((q.c[2] | (q.c[3] << 4)) << 8));
        } else {
          prologue(Ms, nbuf, x, j.eps, lane, y);  // lane holds y[lane + 32u]
          q = quantize(y);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint32_t hi = __shfl_down_sync(0xffffffffu, q.c[u], 1);
            const int byte = (lane + 32 * u) >> 1;  // codes 2 byte, 2 byte + 1
            if ((lane & 1) == 0) dst[16 * ((byte >> 4) ^ k_chunk_swz(slot)) + (byte & 15)] = (uint8_t)(q.c[u] | (hi << 4));
          }
        }
        if (lane == 0) {
          meta[slot] = q.meta;
          if (q.flags) set_err(j.dev_err, q.flags);
        }
      }

      if (!warp_all_finite(xv)) {
        if (lane == 0) set_err(j.dev_err, KVQ_DEVERR_NONFINITE);
      } else {
        const Quant4 q = quantize(xv);  // lane holds elements 4l..4l+3
        const uint32_t two = v_encode4(q.c[0], q.c[1], q.c[2], q.c[3]);
        const int chunk = (lane >> 3) ^ ((slot >> 1) & 3);
        *reinterpret_cast<uint16_t*>(blk + kPage * kRec4 + slot * kRec4 + chunk * 16 + ((2 * lane) & 15)) =
            (uint16_t)two;
        if (lane == 0) {
          meta[kPage + slot] = q.meta;
          if (q.flags) set_err(j.dev_err, q.flags);
        }
      }
    }
  } else {
    const int qb = blockIdx.x - p.kv_blocks, nqb = gridDim.x - p.kv_blocks;
    for (int row = qb * kPrepWarps + warp; row < p.q_jobs; row += nqb * kPrepWarps) {
      float x[4];
      load_row4(j.q, j.q_bf16, (size_t)row, lane, x);
      if (!warp_all_finite(x) && lane == 0) set_err(j.dev_err, KVQ_DEVERR_NONFINITE);
      float y[4];
      if (j.fwht) {  // lane holds q~[4 lane + e]
        prologue_fwht(w4, x, j.eps, lane, y);
        const float4 y4 = make_float4(y[0], y[1], y[2], y[3]);
        reinterpret_cast<float4*>(j.q_rot + (size_t)row * kD)[lane] = y4;
        if (j.q_rot_out) reinterpret_cast<float4*>(j.q_rot_out + (size_t)row * kD)[lane] = y4;
        continue;
      }
      prologue(Ms, nbuf, x, j.eps, lane, y);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        j.q_rot[(size_t)row * kD + lane + 32 * u] = y[u];
        if (j.q_rot_out) j.q_rot_out[(size_t)row * kD + lane + 32 * u] = y[u];
      }
    }
  }
}

// Stock FP8 cache write: one warp per token-head, lane l converts elements 4l..4l+3.
__global__ void fp8_append_kernel(const Fp8AppendJob j) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  const int Hkv = j.ring.num_kv_heads;
  for (int job = warp; job < j.T * Hkv; job += nwarps) {
    const int tok = job / Hkv, h = job - (job / Hkv) * Hkv;
    int seq, pos;
    if (j.seq_ids) {
      seq = j.seq_ids[tok];
      pos = j.positions[tok];
    } else {
      seq = tok / j.S;
      pos = j.pos0[seq] + (tok - seq * j.S);
    }
    if (seq < 0 || seq >= j.ring.num_seqs || pos < 0) {
      if (lane == 0) set_err(j.dev_err, KVQ_DEVERR_POS);
      continue;
    }
    const int slot = pos % j.ring.capacity;
    // block of 64 slots: K records then V records
    uint8_t* blk = j.ring.data + (((size_t)seq * Hkv + h) * (j.ring.capacity / kPage) + slot / kPage) *
                                     (2 * kPage * kRec8);
    for (int which = 0; which < 2; ++which) {
      float x[4];
      load_row4(which ? j.v : j.k, j.bf16, (size_t)tok * Hkv + h, lane, x);
      if (!warp_all_finite(x)) {
        if (lane == 0) set_err(j.dev_err, KVQ_DEVERR_NONFINITE);
        continue;
      }
      fp8_store_row(blk + which * kPage * kRec8, slot, x, which ? j.v_scale : j.k_scale, lane);
    }
  }
}

std::mutex g_prep_mu;  // guards the per-device caches below
int g_sm_count[64] = {0};
bool g_prep_attr[64] = {false};

int sm_count() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  std::lock_guard<std::mutex> lock(g_prep_mu);
  if (g_sm_count[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    g_sm_count[dev] = n > 0 ? n : 1;
  }
  return g_sm_count[dev];
}

}  // namespace

cudaError_t launch_prep(const PrepJobs& jobs, cudaStream_t stream) {
  PrepParams p;
  p.j = jobs;
  p.kv_jobs = jobs.k ? jobs.T * jobs.cache.num_kv_heads : 0;
  p.q_jobs = jobs.q ? jobs.nq_rows : 0;
  if (p.kv_jobs == 0 && p.q_jobs == 0) return cudaSuccess;
  const int cap = 2 * sm_count();
  p.kv_blocks = std::min((p.kv_jobs + kPrepWarps - 1) / kPrepWarps, cap);
  const int q_blocks = std::min((p.q_jobs + kPrepWarps - 1) / kPrepWarps, cap);
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lock(g_prep_mu);
    if (dev < 0 || dev >= 64 || !g_prep_attr[dev]) {
      cudaError_t e = cudaFuncSetAttribute(prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPrepSmem);
      if (e != cudaSuccess) return e;
      if (dev >= 0 && dev < 64) g_prep_attr[dev] = true;
    }
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(p.kv_blocks + q_blocks), 1, 1);
  cfg.blockDim = dim3(kPrepThreads, 1, 1);
  cfg.dynamicSmemBytes = kPrepSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prep_kernel, p);
}

cudaError_t launch_fp8_append(const Fp8AppendJob& job, cudaStream_t stream) {
  const int jobs = job.T * job.ring.num_kv_heads;
  if (jobs == 0) return cudaSuccess;
  const int threads = 256;
  const int blocks = std::min((jobs * 32 + threads - 1) / threads, 4 * sm_count());
  fp8_append_kernel<<<blocks, threads, 0, stream>>>(job);
  return cudaGetLastError();
}

}  // namespace kvq
