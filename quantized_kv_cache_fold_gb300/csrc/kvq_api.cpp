// C-ABI entry points of libkvq: host-side argument checks, the two host-only steps
// (rotation and gain fold) and dispatch to the CUDA kernels. See include/kvq.h for the
// contract of each call.

#include <cmath>
#include <cstdint>
#include <cstring>

#include "kvq.h"
#include "kvq_internal.h"

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

kvq_status from_cuda(cudaError_t e) { return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA; }

// Published splitmix64 step (Steele, Lea, Flood 2014).
uint64_t splitmix64(uint64_t& state) {
  uint64_t z = (state += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

int popcount32(uint32_t x) {
  int c = 0;
  for (; x; x &= x - 1) ++c;
  return c;
}

kvq_status check_int4_cache(const kvq_int4_cache* c) {
  if (!c) return KVQ_ERR_INVALID_ARG;
  if (c->head_dim != KVQ_HEAD_DIM || c->page_size != KVQ_PAGE_SIZE) return KVQ_ERR_UNSUPPORTED;
  if (!c->pages || !c->block_table || !aligned(c->pages, 16)) return KVQ_ERR_INVALID_ARG;
  if (c->num_seqs < 1 || c->max_pages_per_seq < 1 || c->num_pages < 1 || c->num_kv_heads < 1)
    return KVQ_ERR_INVALID_ARG;
  if ((long long)c->max_pages_per_seq * KVQ_PAGE_SIZE > (1LL << 30)) return KVQ_ERR_UNSUPPORTED;
  return KVQ_OK;
}

kvq_status check_ring(const kvq_fp8_ring* r) {
  if (!r) return KVQ_ERR_INVALID_ARG;
  if (r->head_dim != KVQ_HEAD_DIM) return KVQ_ERR_UNSUPPORTED;
  if (!r->data || !aligned(r->data, 16)) return KVQ_ERR_INVALID_ARG;
  if (r->num_seqs < 1 || r->num_kv_heads < 1 || r->capacity < KVQ_PAGE_SIZE || r->capacity % KVQ_PAGE_SIZE)
    return KVQ_ERR_INVALID_ARG;
  return KVQ_OK;
}

bool heads_ok(int Hq, int Hkv, int S) {
  if (Hq < 1 || Hkv < 1 || Hq % Hkv) return false;
  return S * (Hq / Hkv) <= kvq::kMaxRows;
}

}  // namespace

extern "C" {

const char* kvq_status_string(kvq_status s) {
  switch (s) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID_ARG: return "invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "unsupported configuration";
    case KVQ_ERR_CUDA: return "CUDA error";
    case KVQ_ERR_SCRATCH_TOO_SMALL:
      return "request exceeds the fixed scratch of kvq_decode_attn_int4_noalloc (KVQ_NOALLOC_SCRATCH_BYTES)";
  }
  return "unknown status";
}

kvq_status kvq_build_rotation(uint64_t seed, int head_dim, int8_t* s_out, float* R_out) {
  if (head_dim != KVQ_HEAD_DIM) return KVQ_ERR_UNSUPPORTED;
  if (!R_out) return KVQ_ERR_INVALID_ARG;
  int8_t s[KVQ_HEAD_DIM];
  uint64_t st = seed;
  for (int j = 0; j < head_dim; ++j) s[j] = (splitmix64(st) >> 63) ? -1 : 1;
  const double root = std::sqrt((double)head_dim);
  for (int i = 0; i < head_dim; ++i)
    for (int j = 0; j < head_dim; ++j) {
      const int h = (popcount32((uint32_t)(i & j)) & 1) ? -1 : 1;  // Sylvester: (-1)^popcount(i & j)
      R_out[i * head_dim + j] = (float)((double)(h * s[j]) / root);
    }
  if (s_out) std::memcpy(s_out, s, head_dim);
  return KVQ_OK;
}

kvq_status kvq_fold_qk(const float* R, const float* g_q, const float* g_k, int head_dim, float* Mq_out,
                       float* Mk_out) {
  if (head_dim != KVQ_HEAD_DIM) return KVQ_ERR_UNSUPPORTED;
  if (!R || !g_q || !g_k || !Mq_out || !Mk_out) return KVQ_ERR_INVALID_ARG;
  for (int i = 0; i < head_dim; ++i) {
    const double gg = (double)g_q[i] * (double)g_k[i];  // exact in fp64
    for (int j = 0; j < head_dim; ++j) Mq_out[j * head_dim + i] = (float)((double)R[j * head_dim + i] * gg);
  }
  std::memcpy(Mk_out, R, sizeof(float) * head_dim * head_dim);
  return KVQ_OK;
}

kvq_status kvq_fold_qk_fwht(const int8_t* s, const float* g_q, const float* g_k, int head_dim, float* wq_out,
                            float* wk_out) {
  if (head_dim != KVQ_HEAD_DIM) return KVQ_ERR_UNSUPPORTED;
  if (!s || !g_q || !g_k || !wq_out || !wk_out) return KVQ_ERR_INVALID_ARG;
  for (int i = 0; i < head_dim; ++i) {
    if (s[i] != 1 && s[i] != -1) return KVQ_ERR_INVALID_ARG;
    wq_out[i] = (float)((double)s[i] * (double)g_q[i] * (double)g_k[i]);  // exact in fp64, rounded once
    wk_out[i] = (float)s[i];
  }
  return KVQ_OK;
}

static kvq_status append_impl(const kvq_int4_cache* cache, const float* Mk, const void* k, const void* v,
                              kvq_dtype dtype, int T, const int32_t* seq_ids, const int32_t* positions, float eps,
                              int32_t* dev_err, kvq_stream_t stream, int fwht) {
  kvq_status st = check_int4_cache(cache);
  if (st != KVQ_OK) return st;
  if (dtype != KVQ_F32 && dtype != KVQ_BF16) return KVQ_ERR_INVALID_ARG;
  if (T < 0 || (long long)T * cache->num_kv_heads > (1LL << 30)) return KVQ_ERR_INVALID_ARG;
  if (T == 0) return KVQ_OK;
  if (!Mk || !k || !v || !seq_ids || !positions || !dev_err) return KVQ_ERR_INVALID_ARG;
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(Mk, 16)) return KVQ_ERR_INVALID_ARG;
  if (!(eps >= 0.0f) || std::isinf(eps)) return KVQ_ERR_INVALID_ARG;
  kvq::PrepJobs j{};
  j.cache = *cache;
  j.fwht = fwht;
  j.Mk = Mk;
  j.k = k;
  j.v = v;
  j.kv_bf16 = dtype == KVQ_BF16;
  j.T = T;
  j.seq_ids = seq_ids;
  j.positions = positions;
  j.eps = eps;
  j.dev_err = dev_err;
  return from_cuda(kvq::launch_prep(j, (cudaStream_t)stream));
}

kvq_status kvq_rotate_quant_append(const kvq_int4_cache* cache, const float* Mk, const void* k, const void* v,
                                   kvq_dtype dtype, int T, const int32_t* seq_ids, const int32_t* positions,
                                   float eps, int32_t* dev_err, kvq_stream_t stream) {
  return append_impl(cache, Mk, k, v, dtype, T, seq_ids, positions, eps, dev_err, stream, 0);
}

kvq_status kvq_rotate_quant_append_fwht(const kvq_int4_cache* cache, const float* wk, const void* k, const void* v,
                                        kvq_dtype dtype, int T, const int32_t* seq_ids, const int32_t* positions,
                                        float eps, int32_t* dev_err, kvq_stream_t stream) {
  return append_impl(cache, wk, k, v, dtype, T, seq_ids, positions, eps, dev_err, stream, 1);
}

size_t kvq_decode_workspace_bytes(int B, int S, int num_q_heads, int num_kv_heads) {
  if (B < 1 || B > KVQ_MAX_SEQS || S < 1 || S > 8 || !heads_ok(num_q_heads, num_kv_heads, S)) return 0;
  return kvq::workspace_qrot_bytes(B, S, num_q_heads) +
         kvq::workspace_partials_bytes(B, S, num_q_heads, num_kv_heads);
}

}  // extern "C"

namespace kvq {

kvq_status check_decode_int4_args(const kvq_int4_cache* cache, const float* Mq, const float* Mk, const void* q,
                                  kvq_dtype dtype, int B, int S, int num_q_heads, const int32_t* ctx_len,
                                  const void* k_new, const void* v_new, float sm_scale, float eps, const float* out,
                                  const float* q_rot_out, const int32_t* dev_err) {
  kvq_status st = check_int4_cache(cache);
  if (st != KVQ_OK) return st;
  if (S < 1 || S > 8 || !heads_ok(num_q_heads, cache->num_kv_heads, S)) return KVQ_ERR_UNSUPPORTED;
  if (B < 1 || B > KVQ_MAX_SEQS || B > cache->num_seqs) return KVQ_ERR_INVALID_ARG;
  if (dtype != KVQ_F32 && dtype != KVQ_BF16) return KVQ_ERR_INVALID_ARG;
  if (!Mq || !q || !ctx_len || !out || !dev_err) return KVQ_ERR_INVALID_ARG;
  if ((k_new == nullptr) != (v_new == nullptr)) return KVQ_ERR_INVALID_ARG;
  if (k_new && (!Mk || !aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(Mk, 16))) return KVQ_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(Mq, 16)) return KVQ_ERR_INVALID_ARG;
  if (q_rot_out && !aligned(q_rot_out, 16)) return KVQ_ERR_INVALID_ARG;
  if (!std::isfinite(sm_scale) || !(eps >= 0.0f) || std::isinf(eps)) return KVQ_ERR_INVALID_ARG;
  return KVQ_OK;
}

}  // namespace kvq

extern "C" {

static kvq_status decode_int4_impl(const kvq_int4_cache* cache, const float* Mq, const float* Mk, const void* q,
                                   kvq_dtype dtype, int B, int S, int num_q_heads, const int32_t* ctx_len,
                                   const void* k_new, const void* v_new, float sm_scale, float eps, float* out,
                                   void* workspace, size_t workspace_bytes, float* q_rot_out, int32_t* dev_err,
                                   kvq_stream_t stream, int fwht) {
  kvq_status st = kvq::check_decode_int4_args(cache, Mq, Mk, q, dtype, B, S, num_q_heads, ctx_len, k_new, v_new,
                                              sm_scale, eps, out, q_rot_out, dev_err);
  if (st != KVQ_OK) return st;
  if (!workspace || !aligned(workspace, 256)) return KVQ_ERR_INVALID_ARG;
  if (workspace_bytes < kvq_decode_workspace_bytes(B, S, num_q_heads, cache->num_kv_heads))
    return KVQ_ERR_INVALID_ARG;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* q_rot = reinterpret_cast<float*>(ws);
  float* partials = reinterpret_cast<float*>(ws + kvq::workspace_qrot_bytes(B, S, num_q_heads));
  cudaStream_t s = (cudaStream_t)stream;

  kvq::PrepJobs j{};
  j.cache = *cache;
  j.fwht = fwht;
  j.Mk = Mk;
  j.k = k_new;
  j.v = v_new;
  j.kv_bf16 = dtype == KVQ_BF16;
  j.T = k_new ? B * S : 0;
  j.ctx_len = ctx_len;
  j.S = S;
  j.Mq = Mq;
  j.q = q;
  j.q_bf16 = dtype == KVQ_BF16;
  j.nq_rows = B * S * num_q_heads;
  j.q_rot = q_rot;
  j.q_rot_out = q_rot_out;
  j.eps = eps;
  j.dev_err = dev_err;
  cudaError_t e = kvq::launch_prep(j, s);
  if (e != cudaSuccess) return KVQ_ERR_CUDA;

  kvq::AttnJob a{};
  a.fmt = 0;
  a.cache = *cache;
  a.B = B;
  a.S = S;
  a.Hq = num_q_heads;
  a.Hkv = cache->num_kv_heads;
  a.ctx = ctx_len;
  a.q_rot = q_rot;
  a.sm_scale = sm_scale;
  a.out = out;
  a.partials = partials;
  a.dev_err = dev_err;
  return from_cuda(kvq::launch_attention(a, s));
}

kvq_status kvq_decode_attn_int4(const kvq_int4_cache* cache, const float* Mq, const float* Mk, const void* q,
                                kvq_dtype dtype, int B, int S, int num_q_heads, const int32_t* ctx_len,
                                const void* k_new, const void* v_new, float sm_scale, float eps, float* out,
                                void* workspace, size_t workspace_bytes, float* q_rot_out, int32_t* dev_err,
                                kvq_stream_t stream) {
  return decode_int4_impl(cache, Mq, Mk, q, dtype, B, S, num_q_heads, ctx_len, k_new, v_new, sm_scale, eps, out,
                          workspace, workspace_bytes, q_rot_out, dev_err, stream, 0);
}

kvq_status kvq_decode_attn_int4_fwht(const kvq_int4_cache* cache, const float* wq, const float* wk, const void* q,
                                     kvq_dtype dtype, int B, int S, int num_q_heads, const int32_t* ctx_len,
                                     const void* k_new, const void* v_new, float sm_scale, float eps, float* out,
                                     void* workspace, size_t workspace_bytes, float* q_rot_out, int32_t* dev_err,
                                     kvq_stream_t stream) {
  return decode_int4_impl(cache, wq, wk, q, dtype, B, S, num_q_heads, ctx_len, k_new, v_new, sm_scale, eps, out,
                          workspace, workspace_bytes, q_rot_out, dev_err, stream, 1);
}

kvq_status kvq_set_stage_wait_limit_ns(uint64_t ns) {
  kvq::set_stage_wait_limit_ns(ns);
  return KVQ_OK;
}

kvq_status kvq_fp8_swa_plan(int capacity, int B, int S, int num_q_heads, int num_kv_heads, int32_t out[4]) {
  if (!out) return KVQ_ERR_INVALID_ARG;
  if (capacity < KVQ_PAGE_SIZE || capacity % KVQ_PAGE_SIZE || num_kv_heads < 1) return KVQ_ERR_INVALID_ARG;
  if (S < 1 || S > 8 || !heads_ok(num_q_heads, num_kv_heads, S)) return KVQ_ERR_UNSUPPORTED;
  if (B < 1 || B > KVQ_MAX_SEQS) return KVQ_ERR_INVALID_ARG;
  int shape[4];
  kvq::swa_plan_shape(capacity, B, S, num_q_heads, num_kv_heads, shape);
  for (int i = 0; i < 4; ++i) out[i] = shape[i];
  return KVQ_OK;
}

kvq_status kvq_fp8_append(const kvq_fp8_ring* ring, const void* k, const void* v, kvq_dtype dtype, int T,
                          const int32_t* seq_ids, const int32_t* positions, float k_scale, float v_scale,
                          int32_t* dev_err, kvq_stream_t stream) {
  kvq_status st = check_ring(ring);
  if (st != KVQ_OK) return st;
  if (dtype != KVQ_F32 && dtype != KVQ_BF16) return KVQ_ERR_INVALID_ARG;
  if (T < 0 || (long long)T * ring->num_kv_heads > (1LL << 30)) return KVQ_ERR_INVALID_ARG;
  if (T == 0) return KVQ_OK;
  if (!k || !v || !seq_ids || !positions || !dev_err || !aligned(k, 16) || !aligned(v, 16))
    return KVQ_ERR_INVALID_ARG;
  if (!(k_scale > 0.0f) || !(v_scale > 0.0f) || std::isinf(k_scale) || std::isinf(v_scale))
    return KVQ_ERR_INVALID_ARG;
  kvq::Fp8AppendJob j{};
  j.ring = *ring;
  j.k = k;
  j.v = v;
  j.bf16 = dtype == KVQ_BF16;
  j.T = T;
  j.seq_ids = seq_ids;
  j.positions = positions;
  j.k_scale = k_scale;
  j.v_scale = v_scale;
  j.dev_err = dev_err;
  return from_cuda(kvq::launch_fp8_append(j, (cudaStream_t)stream));
}

kvq_status kvq_decode_attn_fp8_swa(const kvq_fp8_ring* ring, const void* q, kvq_dtype dtype, int B, int S,
                                   int num_q_heads, const int32_t* pos0, int window, const void* k_new,
                                   const void* v_new, float k_scale, float v_scale, float sm_scale, float* out,
                                   void* workspace, size_t workspace_bytes, int32_t* dev_err,
                                   kvq_stream_t stream) {
  kvq_status st = check_ring(ring);
  if (st != KVQ_OK) return st;
  if (S < 1 || S > 8 || !heads_ok(num_q_heads, ring->num_kv_heads, S)) return KVQ_ERR_UNSUPPORTED;
  if (B < 1 || B > KVQ_MAX_SEQS || B > ring->num_seqs) return KVQ_ERR_INVALID_ARG;
  if (window < 1 || ring->capacity < window + S - 1) return KVQ_ERR_INVALID_ARG;
  if (dtype != KVQ_F32 && dtype != KVQ_BF16) return KVQ_ERR_INVALID_ARG;
  if (!q || !pos0 || !out || !workspace || !dev_err) return KVQ_ERR_INVALID_ARG;
  if ((k_new == nullptr) != (v_new == nullptr)) return KVQ_ERR_INVALID_ARG;
  if (k_new && (!aligned(k_new, 16) || !aligned(v_new, 16))) return KVQ_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(workspace, 256)) return KVQ_ERR_INVALID_ARG;
  if (!std::isfinite(sm_scale) || !(k_scale > 0.0f) || !(v_scale > 0.0f) || std::isinf(k_scale) ||
      std::isinf(v_scale))
    return KVQ_ERR_INVALID_ARG;
  if (workspace_bytes < kvq_decode_workspace_bytes(B, S, num_q_heads, ring->num_kv_heads))
    return KVQ_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  // Rings that one cluster per (sequence, KV head) covers: one launch that appends the new
  // rows and attends. Larger rings: a separate append, then the split-K path and its combine.
  const bool cluster = kvq::swa_cluster_path(ring->capacity, B, S, num_q_heads, ring->num_kv_heads);
  if (k_new && !cluster) {
    kvq::Fp8AppendJob j{};
    j.ring = *ring;
    j.k = k_new;
    j.v = v_new;
    j.bf16 = dtype == KVQ_BF16;
    j.T = B * S;
    j.pos0 = pos0;
    j.S = S;
    j.k_scale = k_scale;
    j.v_scale = v_scale;
    j.dev_err = dev_err;
    if (kvq::launch_fp8_append(j, s) != cudaSuccess) return KVQ_ERR_CUDA;
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  kvq::AttnJob a{};
  a.fmt = 1;
  a.ring = *ring;
  a.window = window;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.B = B;
  a.S = S;
  a.Hq = num_q_heads;
  a.Hkv = ring->num_kv_heads;
  a.ctx = pos0;
  a.q = q;
  a.q_bf16 = dtype == KVQ_BF16;
  a.k_new = cluster ? k_new : nullptr;
  a.v_new = cluster ? v_new : nullptr;
  a.sm_scale = sm_scale;
  a.out = out;
  a.partials = reinterpret_cast<float*>(ws + kvq::workspace_qrot_bytes(B, S, num_q_heads));
  a.dev_err = dev_err;
  return from_cuda(cluster ? kvq::launch_swa_cluster(a, s) : kvq::launch_attention(a, s));
}

}  // extern "C"
