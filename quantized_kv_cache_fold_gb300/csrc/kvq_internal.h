// Internal launch interface between the C-ABI layer (kvq_api.cpp) and the kernel
// translation units. Host-side only; all arguments have been validated by the caller.
#pragma once

#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "kvq.h"

namespace kvq {

constexpr int kMaxCtas = 1024;       // cap on attention CTAs (sizes the partial-result workspace)
constexpr int kMaxRows = 48;         // S * (num_q_heads / num_kv_heads) rows per KV head and sequence
constexpr int kPartialStride = 130;  // floats per partial row: m, l, acc[128]

// Job description for the prologue/quantise kernel.
struct PrepJobs {
  // int4 append (keys rotated, values raw)
  kvq_int4_cache cache;
  const float* Mk;
  const void* k;
  const void* v;
  int kv_bf16;
  int T;                   // tokens to append (each has num_kv_heads heads)
  const int32_t* seq_ids;  // explicit mode (or null)
  const int32_t* positions;
  const int32_t* ctx_len;  // derived mode: seq = t / S, pos = ctx_len[seq] + t % S
  int S;
  // query prologue
  const float* Mq;
  const void* q;
  int q_bf16;
  int nq_rows;
  float* q_rot;      // workspace destination [nq_rows][128]
  float* q_rot_out;  // optional copy
  float eps;
  int32_t* dev_err;
  // 0: the matrix prologue (Mk, Mq are 128x128 matrices); 1: the FWHT prologue (Mk, Mq are the
  // 128 multipliers w_k = s, w_q = fp32(s g_q g_k) of kvq_fold_qk_fwht)
  int fwht;
};

cudaError_t launch_prep(const PrepJobs& jobs, cudaStream_t stream);

struct Fp8AppendJob {
  kvq_fp8_ring ring;
  const void* k;
  const void* v;
  int bf16;
  int T;
  const int32_t* seq_ids;  // explicit mode (or null)
  const int32_t* positions;
  const int32_t* pos0;     // derived mode: seq = t / S, pos = pos0[seq] + t % S
  int S;
  float k_scale, v_scale;
  int32_t* dev_err;
};

cudaError_t launch_fp8_append(const Fp8AppendJob& job, cudaStream_t stream);

// Attention over either cache format.
struct AttnJob {
  int fmt;  // 0 = int4 paged, 1 = fp8 ring
  kvq_int4_cache cache;
  kvq_fp8_ring ring;
  int window;
  float k_scale, v_scale;
  int B, S, Hq, Hkv;
  const int32_t* ctx;  // int4: ctx_len[b]; fp8: pos0[b]
  const float* q_rot;  // int4: rotated queries [B][S][Hq][128] fp32 (workspace)
  const void* q;       // fp8: queries as given
  int q_bf16;
  const void* k_new;   // fp8 cluster path: rows appended inside the attention kernel (null: none)
  const void* v_new;
  float sm_scale;
  float* out;
  float* partials;  // workspace
  int32_t* dev_err;
};

cudaError_t launch_attention(const AttnJob& job, cudaStream_t stream);

// FP8 window attention with one thread-block cluster per (sequence, KV head), appending
// job.k_new / job.v_new itself. swa_cluster_path() says whether a ring of this capacity, with
// this batch and these head counts, takes it; larger rings go through launch_attention (fmt 1)
// after a separate append.
bool swa_cluster_path(int capacity, int B, int S, int Hq, int Hkv);
// The chosen shape: CTAs per pair (0: split-K path), streams per CTA, stages, units per stream.
void swa_plan_shape(int capacity, int B, int S, int Hq, int Hkv, int out[4]);
cudaError_t launch_swa_cluster(const AttnJob& job, cudaStream_t stream);

// Workspace layout shared by the API and the launchers.
// Host-side argument checks of kvq_decode_attn_int4 other than the workspace (status as that
// call returns it); shared with the allocation-free entry point.
kvq_status check_decode_int4_args(const kvq_int4_cache* cache, const float* Mq, const float* Mk, const void* q,
                                  kvq_dtype dtype, int B, int S, int num_q_heads, const int32_t* ctx_len,
                                  const void* k_new, const void* v_new, float sm_scale, float eps, const float* out,
                                  const float* q_rot_out, const int32_t* dev_err);

// Limit of the split-K attention kernel's stage waits for later launches (kvq_set_stage_wait_limit_ns).
void set_stage_wait_limit_ns(unsigned long long ns);

size_t workspace_qrot_bytes(int B, int S, int Hq);
size_t workspace_partials_bytes(int B, int S, int Hq, int Hkv);

}  // namespace kvq
