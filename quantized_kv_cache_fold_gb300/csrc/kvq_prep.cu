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
// Row stride of the matrix in shared memory, per launch: 132 when passes hold several rows (16-byte
// rows; a 16-byte load of 8 lanes' rows, word offsets 132 j, covers the 32 banks once), 129 when
// every pass is one row (4-byte loads, lanes' rows on distinct banks; fewer wavefronts per load
// than 16-byte loads of one row, the faster form for decode's few rows).
constexpr int kMStride = 132;  // the larger: shared-memory size
// Rows per warp and pass of the matrix prologue (1 to 8, from the call's row counts, see
// launch_prep): each matrix entry read from shared memory serves all of them, and row pairs
// share one fma.rn.f32x2. One row per pass is bound by the matrix reads.
constexpr int kMaxRows = 8;
constexpr int kPrepSmem = (128 * kMStride + kPrepWarps * 128 * kMaxRows) * 4;  // the most a launch asks for
// Shared memory of a launch: the matrix rows and each warp's normalised rows, no more (a prep
// grid starts while the previous grid's blocks still hold shared memory on the SMs).
inline int prep_smem(int mstride, int rows) { return (128 * mstride + kPrepWarps * 128 * rows) * 4; }

struct PrepParams {
  PrepJobs j;
  int kv_blocks;
  int kv_jobs;
  int q_jobs;
  int kv_rows;  // key/value jobs per warp and pass (matrix prologue)
  int q_rows;   // query rows per warp and pass (matrix prologue)
  int mstride;  // row stride of the matrix in shared memory (132, or 129 when both are 1)
  int nrows;    // rows of each warp's normalised-row buffer: max(kv_rows, q_rows)
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

// y[r] = M n(x[r]) for the rows r < nr (rows from nr on are zero and their y is not used).
// Lane l holds x[r][4l..4l+3] and returns y[r][u] = row r's output l + 32u, u = 0..3, each the
// fma chain over k = 0..127 in order, acc = fma(M[l + 32u][k], n[k], acc) from 0, with
// n = fp32(x / sqrt(mean(x^2) + eps)) (norm_inv's order). Rows 2p and 2p + 1 run in the two
// halves of one fma.rn.f32x2, which rounds each half as fma.rn.f32: the chains are unchanged;
// the last row of an odd R > 1 runs as a plain fma.rn.f32 chain in the same order.
// Ms: shared [128][ms], Ms[j ms + k] = M[j][k] (ms = 129 or 132); nbuf: shared float[R][128] of this
// warp (R = 1: n; R > 1: pair p at float 256 p, element k of rows 2p, 2p + 1 side by side, then
// the odd row's n at float 256 (R / 2)).
template <int R>
__device__ __forceinline__ void prologue_rows(const float* __restrict__ Ms, int ms, float* nbuf, const float (&x)[R][4],
                                              int nr, float eps, int lane, float (&y)[R][4]) {
  float nx[R][4];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (r < nr) {
      const float inv = norm_inv(x[r], eps);
#pragma unroll
      for (int e = 0; e < 4; ++e) nx[r][e] = __fmul_rn(x[r][e], inv);
    } else {
      nx[r][0] = nx[r][1] = nx[r][2] = nx[r][3] = 0.0f;
    }
  }
  if constexpr (R == 1) {
    reinterpret_cast<float4*>(nbuf)[lane] = make_float4(nx[0][0], nx[0][1], nx[0][2], nx[0][3]);
  } else {
#pragma unroll
    for (int pr = 0; pr < R / 2; ++pr) {
      float4* d = reinterpret_cast<float4*>(nbuf + pr * 256) + 2 * lane;
      d[0] = make_float4(nx[2 * pr][0], nx[2 * pr + 1][0], nx[2 * pr][1], nx[2 * pr + 1][1]);
      d[1] = make_float4(nx[2 * pr][2], nx[2 * pr + 1][2], nx[2 * pr][3], nx[2 * pr + 1][3]);
    }
    if constexpr ((R & 1) != 0)
      reinterpret_cast<float4*>(nbuf + (R / 2) * 256)[lane] =
          make_float4(nx[R - 1][0], nx[R - 1][1], nx[R - 1][2], nx[R - 1][3]);
  }
  __syncwarp();
  const float* m0 = Ms + lane * ms;
  if constexpr (R == 1) {
    float a[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (ms != kMStride) {  // 4-byte loads (ms = 129)
#pragma unroll 2
      for (int k = 0; k < kD; k += 4) {
        const float4 n4 = reinterpret_cast<const float4*>(nbuf)[k >> 2];
        const float nv[4] = {n4.x, n4.y, n4.z, n4.w};
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int c = 0; c < 4; ++c) a[c] = __fmaf_rn(m0[32 * c * ms + k + u], nv[u], a[c]);
      }
    } else {  // 16-byte loads (ms = 132)
#pragma unroll 2
      for (int k = 0; k < kD; k += 4) {
        const float4 n4 = reinterpret_cast<const float4*>(nbuf)[k >> 2];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float4 m = *reinterpret_cast<const float4*>(m0 + 32 * c * kMStride + k);
          a[c] = __fmaf_rn(m.x, n4.x, a[c]);
          a[c] = __fmaf_rn(m.y, n4.y, a[c]);
          a[c] = __fmaf_rn(m.z, n4.z, a[c]);
          a[c] = __fmaf_rn(m.w, n4.w, a[c]);
        }
      }
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) y[0][c] = a[c];
  } else {
    constexpr int RO = R & 1;  // the odd row's plain chain
    uint64_t a2[R / 2][4];
    float a1[RO + 1][4];
#pragma unroll
    for (int pr = 0; pr < R / 2; ++pr) a2[pr][0] = a2[pr][1] = a2[pr][2] = a2[pr][3] = 0ull;
    a1[0][0] = a1[0][1] = a1[0][2] = a1[0][3] = 0.0f;
#pragma unroll 2
    for (int k = 0; k < kD; k += 4) {
      float4 m[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) m[c] = *reinterpret_cast<const float4*>(m0 + 32 * c * ms + k);
      if constexpr (RO != 0) {
        const float4 n4 = reinterpret_cast<const float4*>(nbuf + (R / 2) * 256)[k >> 2];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          a1[0][c] = __fmaf_rn(m[c].x, n4.x, a1[0][c]);
          a1[0][c] = __fmaf_rn(m[c].y, n4.y, a1[0][c]);
          a1[0][c] = __fmaf_rn(m[c].z, n4.z, a1[0][c]);
          a1[0][c] = __fmaf_rn(m[c].w, n4.w, a1[0][c]);
        }
      }
#pragma unroll
      for (int pr = 0; pr < R / 2; ++pr) {
        const float4 n01 = reinterpret_cast<const float4*>(nbuf + pr * 256)[k >> 1];      // k, k + 1
        const float4 n23 = reinterpret_cast<const float4*>(nbuf + pr * 256)[(k >> 1) + 1];  // k + 2, k + 3
        const uint64_t nn[4] = {f2(n01.x, n01.y), f2(n01.z, n01.w), f2(n23.x, n23.y), f2(n23.z, n23.w)};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          a2[pr][c] = fma_f2(f2(m[c].x, m[c].x), nn[0], a2[pr][c]);
          a2[pr][c] = fma_f2(f2(m[c].y, m[c].y), nn[1], a2[pr][c]);
          a2[pr][c] = fma_f2(f2(m[c].z, m[c].z), nn[2], a2[pr][c]);
          a2[pr][c] = fma_f2(f2(m[c].w, m[c].w), nn[3], a2[pr][c]);
        }
      }
    }
#pragma unroll
    for (int pr = 0; pr < R / 2; ++pr)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        y[2 * pr][c] = f2lo(a2[pr][c]);
        y[2 * pr + 1][c] = f2hi(a2[pr][c]);
      }
    if constexpr (RO != 0)
#pragma unroll
      for (int c = 0; c < 4; ++c) y[R - 1][c] = a1[0][c];
  }
  __syncwarp();
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

// Page block and slot of key/value job `job` (token-head, row index token * Hkv + head), or
// nullptr after recording the error (position outside the sequence's pages, or a block-table
// entry outside the pool).
__device__ __forceinline__ uint8_t* job_block(const PrepJobs& j, int job, int lane, int& slot) {
  const int Hkv = j.cache.num_kv_heads;
  const int tok = job / Hkv, h = job - (job / Hkv) * Hkv;
  int seq, pos;
  if (j.seq_ids) {
    seq = j.seq_ids[tok];
    pos = j.positions[tok];
  } else {
    seq = tok / j.S;
    pos = j.ctx_len[seq] + (tok - seq * j.S);
  }
  slot = 0;
  if (seq < 0 || seq >= j.cache.num_seqs || pos < 0 || pos >= j.cache.max_pages_per_seq * kPage) {
    if (lane == 0) set_err(j.dev_err, KVQ_DEVERR_POS);
    return nullptr;
  }
  const int page = j.cache.block_table[(size_t)seq * j.cache.max_pages_per_seq + pos / kPage];
  if (page < 0 || page >= j.cache.num_pages) {
    if (lane == 0) set_err(j.dev_err, KVQ_DEVERR_PAGE);
    return nullptr;
  }
  slot = pos & (kPage - 1);
  return j.cache.pages + ((size_t)page * Hkv + h) * KVQ_INT4_BLOCK_BYTES;
}

// Stores one job's key codes qk (matrix prologue order: lane holds outputs lane + 32u; FWHT
// order: 4 lane + e) and value codes qv with their scales and offsets into slot `slot` of
// block `blk`; a row that held a non-finite value is skipped and recorded instead.
__device__ __forceinline__ void store_job(const PrepJobs& j, uint8_t* blk, int slot, bool k_finite, bool v_finite,
                                          const Quant4& qk, const Quant4& qv, bool fwht_order, int lane) {
  uint32_t* meta = reinterpret_cast<uint32_t*>(blk + 2 * kPage * kRec4);
  if (!k_finite) {
    if (lane == 0) set_err(j.dev_err, KVQ_DEVERR_NONFINITE);
  } else {
    uint8_t* dst = blk + slot * kRec4;
    if (fwht_order) {  // codes 4l..4l+3 = bytes 2l, 2l+1
      *reinterpret_cast<uint16_t*>(dst + 16 * ((lane >> 3) ^ k_chunk_swz(slot)) + ((2 * lane) & 15)) =
          (uint16_t)((qk.c[0] | (qk.c[1] << 4)) | ((qk.c[2] | (qk.c[3] << 4)) << 8));
    } else {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t hi = __shfl_down_sync(0xffffffffu, qk.c[u], 1);
        const int byte = (lane + 32 * u) >> 1;  // codes 2 byte, 2 byte + 1
        if ((lane & 1) == 0) dst[16 * ((byte >> 4) ^ k_chunk_swz(slot)) + (byte & 15)] = (uint8_t)(qk.c[u] | (hi << 4));
      }
    }
    if (lane == 0) {
      meta[slot] = qk.meta;
      if (qk.flags) set_err(j.dev_err, qk.flags);
    }
  }
  if (!v_finite) {
    if (lane == 0) set_err(j.dev_err, KVQ_DEVERR_NONFINITE);
  } else {
    const uint32_t two = v_encode4(qv.c[0], qv.c[1], qv.c[2], qv.c[3]);  // lane holds elements 4l..4l+3
    const int chunk = (lane >> 3) ^ ((slot >> 1) & 3);
    *reinterpret_cast<uint16_t*>(blk + kPage * kRec4 + slot * kRec4 + chunk * 16 + ((2 * lane) & 15)) = (uint16_t)two;
    if (lane == 0) {
      meta[kPage + slot] = qv.meta;
      if (qv.flags) set_err(j.dev_err, qv.flags);
    }
  }
}

// Key/value jobs of this block with the matrix prologue, R consecutive jobs per warp and pass.
// Every row of a pass is loaded, and every job's slot looked up, before any is used; the pass's
// key and value rows are quantised with no store in between (their shuffle and division chains
// interleave), then stored.
template <int R>
__device__ __forceinline__ void kv_rows_matrix(const PrepParams& p, const float* Ms, float* nbuf, int warp, int lane) {
  const PrepJobs& j = p.j;
  for (int job0 = ((int)blockIdx.x * kPrepWarps + warp) * R; job0 < p.kv_jobs; job0 += p.kv_blocks * kPrepWarps * R) {
    const int nr = min(R, p.kv_jobs - job0);
    float x[R][4], xv[R][4], y[R][4];
    uint8_t* blk[R];
    int slot[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (r < nr) {
        load_row4(j.k, j.kv_bf16, (size_t)(job0 + r), lane, x[r]);
        load_row4(j.v, j.kv_bf16, (size_t)(job0 + r), lane, xv[r]);
      } else {
        x[r][0] = x[r][1] = x[r][2] = x[r][3] = 0.0f;
        xv[r][0] = xv[r][1] = xv[r][2] = xv[r][3] = 0.0f;
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) blk[r] = r < nr ? job_block(j, job0 + r, lane, slot[r]) : nullptr;
    bool kf[R], vf[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      kf[r] = warp_all_finite(x[r]);
      vf[r] = warp_all_finite(xv[r]);
    }
    prologue_rows<R>(Ms, p.mstride, nbuf, x, nr, j.eps, lane, y);
    Quant4 qk[R], qv[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      qk[r] = quantize(y[r]);
      qv[r] = quantize(xv[r]);
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
      if (blk[r]) store_job(j, blk[r], slot[r], kf[r], vf[r], qk[r], qv[r], false, lane);
  }
}

// Query rows of this block with the matrix prologue, R rows per warp and pass. Every row of a
// pass is loaded before any is checked, so the loads are in flight together.
template <int R>
__device__ __forceinline__ void q_rows_matrix(const PrepParams& p, const float* Ms, float* nbuf, int qb, int nqb,
                                              int warp, int lane) {
  const PrepJobs& j = p.j;
  for (int row0 = (qb * kPrepWarps + warp) * R; row0 < p.q_jobs; row0 += nqb * kPrepWarps * R) {
    const int nr = min(R, p.q_jobs - row0);
    float x[R][4], y[R][4];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (r < nr) {
        load_row4(j.q, j.q_bf16, (size_t)(row0 + r), lane, x[r]);
      } else {
        x[r][0] = x[r][1] = x[r][2] = x[r][3] = 0.0f;
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
      if (r < nr && !warp_all_finite(x[r]) && lane == 0) set_err(j.dev_err, KVQ_DEVERR_NONFINITE);
    prologue_rows<R>(Ms, p.mstride, nbuf, x, nr, j.eps, lane, y);  // lane holds y[r][lane + 32u]
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (r < nr) {
        const size_t row = (size_t)(row0 + r);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          j.q_rot[row * kD + lane + 32 * u] = y[r][u];
          if (j.q_rot_out) j.q_rot_out[row * kD + lane + 32 * u] = y[r][u];
        }
      }
    }
  }
}

// RQ: query rows per warp and pass, RKV: key/value jobs per warp and pass (at most 4: a pass holds
// key, value and output rows), with the matrix prologue; one of each with the FWHT one. One
// instantiation per shape keeps each launch's code to its own path (the decode launch, 1 and 1,
// is a short latency-bound grid).
template <int RQ, int RKV>
__global__ void __launch_bounds__(kPrepThreads, 2) prep_kernel(const PrepParams p) {
  static_assert(RQ >= 1 && RQ <= kMaxRows && RKV >= 1 && RKV <= 4, "prep pass shapes");
  extern __shared__ __align__(16) float smem_f[];
  float* Ms = smem_f;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* nbuf = smem_f + 128 * p.mstride + warp * 128 * p.nrows;
  const PrepJobs& j = p.j;
  const bool kv_role = (int)blockIdx.x < p.kv_blocks;
  const float* M = kv_role ? j.Mk : j.Mq;
  // May overlap the previous grid on the stream. Before the wait: L2 prefetches of this warp's
  // first rows, and the folded weights (M, or the FWHT multipliers), which are complete before
  // the call (kvq.h) and are staged into shared memory now.
  const size_t rbytes = (size_t)kD * ((kv_role ? j.kv_bf16 : j.q_bf16) ? 2 : 4);
  // rows per warp and pass: p.kv_rows / p.q_rows with the matrix prologue, one with the FWHT one
  const int nrows = j.fwht ? 1 : (kv_role ? p.kv_rows : p.q_rows);
  const int job0 = kv_role ? ((int)blockIdx.x * kPrepWarps + warp) * nrows
                           : (((int)blockIdx.x - p.kv_blocks) * kPrepWarps + warp) * nrows;
  const int njobs = kv_role ? p.kv_jobs : p.q_jobs;
  const bool has_job0 = job0 < njobs;
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
  const int n0 = has_job0 ? min(nrows, njobs - job0) : 1;  // the first pass's rows are consecutive
  if (lane == 0 && r0a) prefetch_l2_bulk(r0a, (uint32_t)(rbytes * n0));
  if (lane == 0 && r0b) prefetch_l2_bulk(r0b, (uint32_t)(rbytes * n0));
  // the FWHT prologue needs only this lane's four multipliers; the matrix prologue stages M
  const float4 w4 = j.fwht ? reinterpret_cast<const float4*>(M)[lane] : make_float4(0.f, 0.f, 0.f, 0.f);
  if (!j.fwht) {
    // 16 independent 16-byte loads per thread, then the shared stores into padded rows
    constexpr int kPer = kD * kD / 4 / kPrepThreads;
    float4 v[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) v[u] = reinterpret_cast<const float4*>(M)[threadIdx.x + u * kPrepThreads];
    const int ms = p.mstride;
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int e = 4 * (threadIdx.x + u * kPrepThreads);
      float* d = Ms + (e >> 7) * ms + (e & 127);
      if (ms == kMStride) {
        *reinterpret_cast<float4*>(d) = v[u];
      } else {
        d[0] = v[u].x;
        d[1] = v[u].y;
        d[2] = v[u].z;
        d[3] = v[u].w;
      }
    }
  }
  __syncthreads();
  griddep_wait();
  griddep_launch_dependents();

  if (kv_role) {
    if (j.fwht) {
      for (int job = blockIdx.x * kPrepWarps + warp; job < p.kv_jobs; job += p.kv_blocks * kPrepWarps) {
        float x[1][4], xv[1][4];
        load_row4(j.k, j.kv_bf16, (size_t)job, lane, x[0]);  // row index = token * Hkv + head = job
        load_row4(j.v, j.kv_bf16, (size_t)job, lane, xv[0]);
        float y[4];
        prologue_fwht(w4, x[0], j.eps, lane, y);  // lane holds y[4 lane + e]
        int slot;
        uint8_t* blk = job_block(j, job, lane, slot);
        if (blk)
          store_job(j, blk, slot, warp_all_finite(x[0]), warp_all_finite(xv[0]), quantize(y), quantize(xv[0]), true,
                    lane);
      }
      return;
    }
    kv_rows_matrix<RKV>(p, Ms, nbuf, warp, lane);
  } else {
    const int qb = blockIdx.x - p.kv_blocks, nqb = gridDim.x - p.kv_blocks;
    if (j.fwht) {
      for (int row = qb * kPrepWarps + warp; row < p.q_jobs; row += nqb * kPrepWarps) {
        float x[4], y[4];
        load_row4(j.q, j.q_bf16, (size_t)row, lane, x);
        if (!warp_all_finite(x) && lane == 0) set_err(j.dev_err, KVQ_DEVERR_NONFINITE);
        prologue_fwht(w4, x, j.eps, lane, y);  // lane holds q~[4 lane + e]
        const float4 y4 = make_float4(y[0], y[1], y[2], y[3]);
        reinterpret_cast<float4*>(j.q_rot + (size_t)row * kD)[lane] = y4;
        if (j.q_rot_out) reinterpret_cast<float4*>(j.q_rot_out + (size_t)row * kD)[lane] = y4;
      }
      return;
    }
    q_rows_matrix<RQ>(p, Ms, nbuf, qb, nqb, warp, lane);
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
// Pass shapes (query rows, key/value jobs per warp and pass) of the matrix prologue's
// instantiations; the FWHT prologue takes the first.
struct PrepShape {
  int rq, rkv;
  const void* kern;
};
const PrepShape kPrepShapes[] = {
    {1, 1, (const void*)prep_kernel<1, 1>}, {2, 1, (const void*)prep_kernel<2, 1>},
    {2, 2, (const void*)prep_kernel<2, 2>}, {3, 2, (const void*)prep_kernel<3, 2>},
    {4, 2, (const void*)prep_kernel<4, 2>}, {4, 3, (const void*)prep_kernel<4, 3>},
    {6, 3, (const void*)prep_kernel<6, 3>}, {6, 4, (const void*)prep_kernel<6, 4>},
    {8, 4, (const void*)prep_kernel<8, 4>},
};
constexpr int kNumPrepShapes = (int)(sizeof(kPrepShapes) / sizeof(kPrepShapes[0]));
bool g_prep_attr[64][kNumPrepShapes] = {{false}};  // per device and instantiation

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

// Work of a key/value job against a query row in the matrix prologue: the same matrix product,
// plus two quantisations (the key's and the value's), the row loads and the slot look-up;
// measured per block on 64 x 16,384 tokens at S = 8 (4 jobs per warp 14.5 us, 6 query rows per
// warp 11.3 us): about 2.
constexpr double kKvWeight = 2.0;

// Largest work (query rows, key/value jobs weighted kKvWeight) that one SM receives from a grid
// of kvb key/value blocks then qb query blocks, dealt round robin over sm SMs (block i shares
// an SM with block i + sm), each warp taking rkv jobs or rq rows; the matrix product makes the
// kernel bound by the SM's FMA throughput once several passes share it.
double prep_sm_load(long long kv_jobs, long long q_jobs, int kvb, int qb, int rkv, int rq, int sm) {
  auto block_load = [&](long long i) -> double {
    if (i < kvb) return kKvWeight * (double)std::min<long long>(kPrepWarps * rkv, kv_jobs - i * kPrepWarps * rkv);
    i -= kvb;
    return (double)std::min<long long>(kPrepWarps * rq, q_jobs - i * kPrepWarps * rq);
  };
  const long long n = (long long)kvb + qb;
  double worst = 0.0;
  for (long long s = 0; s < std::min<long long>(n, sm); ++s)
    worst = std::max(worst, block_load(s) + (s + sm < n ? block_load(s + sm) : 0.0));
  return worst;
}

}  // namespace

cudaError_t launch_prep(const PrepJobs& jobs, cudaStream_t stream) {
  PrepParams p;
  p.j = jobs;
  p.kv_jobs = jobs.k ? jobs.T * jobs.cache.num_kv_heads : 0;
  p.q_jobs = jobs.q ? jobs.nq_rows : 0;
  if (p.kv_jobs == 0 && p.q_jobs == 0) return cudaSuccess;
  const int sm = sm_count();
  const int cap = 2 * sm;  // one wave: two blocks per SM (shared memory)
  int shape = 0, q_blocks = 0;
  if (jobs.fwht) {
    // one row per warp and pass; blocks shared between the roles in proportion to work
    const int kv_max = (p.kv_jobs + kPrepWarps - 1) / kPrepWarps, q_max = (p.q_jobs + kPrepWarps - 1) / kPrepWarps;
    if (kv_max + q_max <= cap) {
      p.kv_blocks = kv_max;
      q_blocks = q_max;
    } else {
      const double wkv = kKvWeight * p.kv_jobs, wq = p.q_jobs;
      p.kv_blocks = std::min(kv_max, std::max(p.kv_jobs ? 1 : 0, (int)(cap * wkv / (wkv + wq) + 0.5)));
      q_blocks = std::min(q_max, std::max(p.q_jobs ? 1 : 0, cap - p.kv_blocks));
    }
  } else {
    // the pass shape whose grid (one pass per warp) fits one wave with the least work on any SM,
    // then the fewest rows per pass (a pass's latency grows with its rows); calls too large for
    // one wave take the largest shape, several passes per warp, blocks shared in proportion to work
    double best = 0.0;
    shape = -1;
    for (int i = 0; i < kNumPrepShapes; ++i) {
      const int rq = kPrepShapes[i].rq, rkv = kPrepShapes[i].rkv;
      const int kvb = (p.kv_jobs + kPrepWarps * rkv - 1) / (kPrepWarps * rkv);
      const int qb = (p.q_jobs + kPrepWarps * rq - 1) / (kPrepWarps * rq);
      if (kvb + qb > cap) continue;
      const double load = prep_sm_load(p.kv_jobs, p.q_jobs, kvb, qb, rkv, rq, sm);
      if (shape < 0 || load < best) {
        best = load;
        shape = i;
        p.kv_blocks = kvb;
        q_blocks = qb;
      }
    }
    if (shape < 0) {
      shape = kNumPrepShapes - 1;
      const int rq = kPrepShapes[shape].rq, rkv = kPrepShapes[shape].rkv;
      const int kv_max = (p.kv_jobs + kPrepWarps * rkv - 1) / (kPrepWarps * rkv);
      const int q_max = (p.q_jobs + kPrepWarps * rq - 1) / (kPrepWarps * rq);
      const double wkv = kKvWeight * p.kv_jobs, wq = p.q_jobs;
      p.kv_blocks = std::min(kv_max, std::max(p.kv_jobs ? 1 : 0, (int)(cap * wkv / (wkv + wq) + 0.5)));
      q_blocks = std::min(q_max, std::max(p.q_jobs ? 1 : 0, cap - p.kv_blocks));
    }
  }
  p.q_rows = kPrepShapes[shape].rq;
  p.kv_rows = kPrepShapes[shape].rkv;
  p.mstride = p.kv_rows == 1 && p.q_rows == 1 ? 129 : kMStride;
  p.nrows = std::max(p.kv_rows, p.q_rows);
  const void* kern = kPrepShapes[shape].kern;
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lock(g_prep_mu);
    if (dev < 0 || dev >= 64 || !g_prep_attr[dev][shape]) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kPrepSmem);
      if (e != cudaSuccess) return e;
      if (dev >= 0 && dev < 64) g_prep_attr[dev][shape] = true;
    }
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(p.kv_blocks + q_blocks), 1, 1);
  cfg.blockDim = dim3(kPrepThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)prep_smem(p.mstride, p.nrows);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {&p};
  return cudaLaunchKernelExC(&cfg, kern, args);
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
