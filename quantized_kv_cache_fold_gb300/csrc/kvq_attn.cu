// Split-K flash-decoding attention over the rotated int4 cache and the FP8 ring.
//
// "Serving Kolibri-1 with a 4-bit KV cache", section "What we do": decode reads the 4-bit
// codes directly and nothing is rotated back. Sliding-window layers whose FP8 ring is too
// large for one thread-block cluster per (sequence, KV head) (kvq_swa.cu) read it through
// the same kernel (FMT = 1).
//
// Work split (stream-K over pages): every (sequence b, KV head h) is a segment of np_b
// pages; the segments are laid end to end and each CTA takes an equal contiguous range of
// pages, so ragged contexts balance to within one page. A CTA emits one partial
// (m, l, acc[128] per query row) for every segment it touches, into slot cta + segment;
// combine_kernel merges a segment's partials with log-sum-exp weights.
//
// Inside a CTA: one producer warp streams page-head blocks (K codes, V codes, K/V meta)
// into a ring of shared-memory stages with bulk asynchronous copies (TMA engine) signalled
// on mbarriers; consumer warps are arranged as token groups x tile groups. A tile is 8
// query rows (rows = S x G query heads of the KV head, row n = r*G + g). Per page a warp:
//   QK^T on tensor cores (mma.m16n8k16, fp32 accumulate): A = 16 tokens x 16 dims of K codes
//        read as the f16 subnormals c 2^-24 (low nibbles) or 16c 2^-24 (high nibbles, whose
//        query values are divided by 16), B = 16 dims x 8 query rows of q~ in f16, so the
//        accumulator holds 2^-24 sum q~ c up to fp32 rounding;
//   score = log2(e)*sm_scale*(s_K*dot + o_K*sum(q~)) -- scale and offset per token;
//   online softmax with exp2 against a lazily moved base (moved only when a score passes it
//        by more than 8, or by anything on pages with a V scale of 255 or more);
//   PV on tensor cores: A = 16 dims x 16 tokens of V codes read as f16 subnormals
//        (c - 7.5) 2^(k - 23), exact and centred (which keeps the fp32 sums of long contexts
//        small), B = 16 tokens x 8 rows of p*s_V in f16 (movmatrix transposes the QK
//        accumulator), plus sum_j p_j (o_V + 7.5 s_V) added per row; the partial undoes
//        2^(k - 23) per dim.

#include <algorithm>
#include <cmath>

#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

// Tuning of the attention CTA when one warp covers every query row of a KV head (S*G <= 8):
// consumer token groups, shared-memory pipeline stages and the register cap per thread.
#ifndef KVQ_TOKEN_GROUPS
#define KVQ_TOKEN_GROUPS 4
#endif
#ifndef KVQ_STAGES_INT4
#define KVQ_STAGES_INT4 12
#endif
#ifndef KVQ_INT4_MAXREG
#define KVQ_INT4_MAXREG 168
#endif
// int4 split kernel with 2 or 3 row tiles in one warp (one CTA per SM: about 250 registers a
// thread): 7 token groups, so 8 warps, two per SM sub-partition (4 -> 7: 300 -> 248 us at S = 2
// on the 64k workload), and 14 stages.
#ifndef KVQ_TILES3_TOKEN_GROUPS
#define KVQ_TILES3_TOKEN_GROUPS 7
#endif
#ifndef KVQ_TILES3_STAGES
#define KVQ_TILES3_STAGES 14
#endif
// 4 to 6 row tiles: two tile groups of up to 3 tiles, 3 token groups (7 warps), 6 stages.
#ifndef KVQ_TILES6_TOKEN_GROUPS
#define KVQ_TILES6_TOKEN_GROUPS 3
#endif
#ifndef KVQ_TILES6_STAGES
#define KVQ_TILES6_STAGES 6
#endif
// A consumer warp takes pages kg, kg + nkg, ... and page k lands in stage k mod nstages with
// phase parity (k / nstages) & 1. Parity only tells adjacent phases apart, so every stage
// must belong to one consumer warp (nstages a multiple of nkg); otherwise a warp running
// ahead could pass the wait for round f while round f - 1 of that stage is still in flight.
static_assert(KVQ_STAGES_INT4 % KVQ_TOKEN_GROUPS == 0, "stages must be a multiple of the token groups");

constexpr int kStage4 = 2 * kPage * kRec4 + 2 * kPage * 4;  // 8704 bytes: K codes, V codes, K meta, V meta
constexpr int kStage8 = 2 * kPage * kRec8;                  // 16384 bytes: K and V e4m3
constexpr float kLog2e = 1.4426950408889634f;

struct AttnParams {
  // int4: page-head blocks [num_pages][Hkv][8704]; fp8: ring blocks [B][Hkv][cap/64][16384]
  const uint8_t* blocks;
  const int32_t* block_table;
  int max_pages;
  int num_pages;
  // fp8 ring
  int cap;
  int window;
  float v_scale;
  // shape
  int B, S, Hq, Hkv, G, R;
  const int32_t* ctx;
  const float* q_rot;
  const void* q;
  int q_bf16;
  float score_scale;
  float* partials;
  float* out;
  int32_t* dev_err;
  int ntg, nkg, nstages, rows_pad;
  int n_cta;
  // limit of the split kernel's waits on its shared-memory stages (consumers on a page's
  // copy, the producer on a stage's release); the drain of copies in flight keeps kWaitLimitNs
  unsigned long long stage_wait_ns;
};

__host__ __device__ __forceinline__ size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Per-lane online-softmax state of one 8-row tile as the token groups exchange it at a
// segment end: m and l and ov of the lane's two rows, then its 32 accumulator values.
constexpr int kMergeFloats = 6 + 32;

// Shared-memory layout, identical on host (sizing) and device.
struct SmemLayout {
  size_t stages, full, empty, valid, red, pre, flags, total;
  __host__ __device__ SmemLayout(int fmt, int nstages, int B, int nkg, int rows_pad) {
    const size_t stage = fmt == 0 ? kStage4 : kStage8;
    stages = 0;
    full = align_up(stages + nstages * stage, 16);
    empty = full + 8 * nstages;
    valid = empty + 8 * nstages;
    red = align_up(valid + 4 * nstages, 16);
    // one merge slot per tile group: kMergeFloats floats per lane per 8-row tile (lane-major)
    pre = align_up(red + (size_t)(rows_pad / 8) * kMergeFloats * 32 * 4, 128);
    flags = pre + 4 * (B + 1);
    total = align_up(flags + 16, 16);
  }
};

// Context length of sequence b as used by every kernel of one call (clamped into the
// cache; `bad` reports a clamp). Read at L2 (ld.global.cg): combine_kernel reads it before
// waiting for the previous grid, so no line an SM's L1 kept from an earlier call may serve it.
__device__ __forceinline__ int eff_ctx(const AttnParams& p, int b, bool& bad, int fmt) {
  int c = __ldcg(p.ctx + b);
  if (fmt == 0) {
    const int cap = p.max_pages * kPage - p.S;
    if (c < 0 || c > cap) {
      bad = true;
      c = min(max(c, 0), cap);
    }
  } else if (c < 0) {
    bad = true;
    c = 0;
  }
  return c;
}

__device__ __forceinline__ int seg_pages(const AttnParams& p, int ctxb, int fmt) {
  return fmt == 0 ? (ctxb + p.S + kPage - 1) / kPage : p.cap / kPage;
}

// Warp 0 builds pre[b] = sum_{b' < b} np_b' (pre[B] = total pages per KV head) and
// flags[1] = any clamped context. Other warps return at once.
__device__ void build_prefix(const AttnParams& p, int fmt, int* pre, volatile int* flags) {
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  if (fmt == 1) {  // every window segment spans the whole ring: no context lengths needed
    const int nblk = p.cap / kPage;
    for (int b = lane; b <= p.B; b += 32) pre[b] = b * nblk;
    if (lane == 0) {
      flags[0] = 0;
      flags[1] = 0;
    }
    return;
  }
  int carry = 0;
  bool bad = false;
  for (int base = 0; base < p.B; base += 32) {
    const int b = base + lane;
    int np = 0;
    if (b < p.B) np = seg_pages(p, eff_ctx(p, b, bad, fmt), fmt);
    int incl = np;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (b < p.B) pre[b] = carry + incl - np;
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  const bool any_bad = __any_sync(0xffffffffu, bad);
  if (lane == 0) {
    pre[p.B] = carry;
    flags[0] = 0;
    flags[1] = any_bad ? 1 : 0;
  }
}

// Flattened page -> (sequence, head, local page, pages of the sequence).
__device__ __forceinline__ void decode_page(const int* pre, int B, int Hkv, long long pg, int& b, int& h, int& lp,
                                            int& np) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((long long)Hkv * pre[mid] <= pg)
      lo = mid;
    else
      hi = mid - 1;
  }
  b = lo;
  np = pre[b + 1] - pre[b];
  const long long rem = pg - (long long)Hkv * pre[b];
  h = (int)(rem / np);
  lp = (int)(rem - (long long)h * np);
}

// CTA whose page range [floor(i P / n), floor((i+1) P / n)) contains page pg (n <= P).
__device__ __forceinline__ long long cta_of(long long pg, long long P, int n) { return ((pg + 1) * n - 1) / P; }

__device__ __forceinline__ float h2f_lo(uint32_t x) {
  return __half2float(__ushort_as_half((unsigned short)(x & 0xFFFFu)));
}
__device__ __forceinline__ float h2f_hi(uint32_t x) { return __half2float(__ushort_as_half((unsigned short)(x >> 16))); }

// Output dim of accumulator row `row` (0..15) of PV m-tile `mt` (0..7).
template <int FMT>
__device__ __forceinline__ int out_dim(int mt, int row) {
  if (FMT == 0) return 32 * (mt >> 1) + 4 * (row & 7) + 2 * (mt & 1) + (row >> 3);
  return 16 * mt + 2 * (row & 7) + (row >> 3);
}

// Producer warp of the split kernels: the 32 lanes resolve the source blocks of 32 consecutive
// pages of the CTA's range [p0, p1) at once (block-table loads in parallel); lane 0 then issues
// one bulk copy per page into the ring of `nst` stages, in order, as stages free (`empty`, one
// phase per round), signalling `full`. A page whose block-table entry is out of range is
// flagged and delivered as invalid (valid[s] = 0, no copy). Waits for its own copies before
// returning.
template <int FMT>
__device__ __forceinline__ void produce_pages(const AttnParams& p, const int* pre, uint8_t* stages, uint64_t* full,
                                              uint64_t* empty, volatile int* valid, volatile int* flags, int nst,
                                              long long p0, long long p1, int lane) {
  constexpr int kStage = FMT == 0 ? kStage4 : kStage8;
  const uint64_t pol = policy_evict_first();
  const int npages = (int)(p1 - p0);
  int issued = 0;
  int s = 0, f = 0;  // stage and fill round of the next page
  for (int base = 0; base < npages; base += 32) {
    const int mine = base + lane;
    long long src = -1;  // byte offset of the page's block; -1 = invalid page
    if (mine < npages) {
      int b, h, lp, np;
      decode_page(pre, p.B, p.Hkv, p0 + mine, b, h, lp, np);
      if (FMT == 0) {
        const int phys = p.block_table[(size_t)b * p.max_pages + lp];
        if (phys >= 0 && phys < p.num_pages)
          src = ((long long)phys * p.Hkv + h) * kStage4;
        else
          set_err(p.dev_err, KVQ_DEVERR_PAGE);
      } else {
        src = (((long long)b * p.Hkv + h) * (p.cap / kPage) + lp) * kStage8;
      }
    }
    const int n = min(32, npages - base);
    int halt = 0;
    for (int j = 0; j < n; ++j) {
      const long long sj = __shfl_sync(0xffffffffu, src, j);
      if (lane == 0 && !halt) {
        if (f > 0 && !mbar_wait_bounded(&empty[s], (f - 1) & 1, p.stage_wait_ns)) {
          set_err(p.dev_err, KVQ_DEVERR_TIMEOUT);
          flags[0] = 1;
          halt = 1;
        } else {
          if (sj < 0) {
            valid[s] = 0;
            mbar_arrive(&full[s]);
          } else {
            valid[s] = 1;
            mbar_arrive_expect_tx(&full[s], kStage);
            bulk_g2s(stages + (size_t)s * kStage, p.blocks + sj, kStage, &full[s], pol);
          }
          ++issued;
          if (++s == nst) {
            s = 0;
            ++f;
          }
        }
      }
    }
    if (__shfl_sync(0xffffffffu, halt | flags[0], 0)) break;
  }
  // Do not retire while copies into this CTA's shared memory may be in flight.
  if (lane == 0) {
    for (int st = 0; st < nst && st < issued; ++st) {
      const int last = st + ((issued - 1 - st) / nst) * nst;
      if (!mbar_wait_bounded(&full[st], (last / nst) & 1)) set_err(p.dev_err, KVQ_DEVERR_TIMEOUT);
    }
  }
}

// Register caps: the int4 single-tile CTA (5 warps) must fit twice per SM, i.e. 3 warps per
// SM sub-partition -> at most 170 registers.
template <int FMT, int NT>
__global__ void __maxnreg__(NT == 1 ? (FMT == 0 ? KVQ_INT4_MAXREG : 184) : 255)
    attn_kernel(const AttnParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int kStage = FMT == 0 ? kStage4 : kStage8;
  constexpr int MTU = NT == 1 ? 4 : 2;  // 16-token m-tiles per online-softmax update
  const SmemLayout L(FMT, p.nstages, p.B, p.nkg, p.rows_pad);
  uint8_t* stages = smem + L.stages;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.full);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.empty);
  volatile int* valid = reinterpret_cast<volatile int*>(smem + L.valid);
  int* pre = reinterpret_cast<int*>(smem + L.pre);
  volatile int* flags = reinterpret_cast<volatile int*>(smem + L.flags);
  float* red = reinterpret_cast<float*>(smem + L.red);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwc = p.ntg * p.nkg;
  const int nst = p.nstages;

  // launched with programmatic serialisation: nothing is read before the previous grid is done
  griddep_wait();
  griddep_launch_dependents();
  build_prefix(p, FMT, pre, flags);
  if (threadIdx.x < nst) {
    mbar_init(&full[threadIdx.x], 1);
    mbar_init(&empty[threadIdx.x], p.ntg);
  }
  fence_barrier_init();
  __syncthreads();

  if (blockIdx.x == 0 && threadIdx.x == 0 && flags[1]) set_err(p.dev_err, KVQ_DEVERR_POS);
  const long long P = (long long)p.Hkv * pre[p.B];
  const int n_eff = (int)min((long long)p.n_cta, P);
  if ((int)blockIdx.x >= n_eff) return;
  const long long p0 = (long long)blockIdx.x * P / n_eff;
  const long long p1 = (long long)(blockIdx.x + 1) * P / n_eff;

  // ------------------------------------------------------------ producer warp
  if (warp == nwc) {
    produce_pages<FMT>(p, pre, stages, full, empty, valid, flags, nst, p0, p1, lane);
    return;
  }

  // ------------------------------------------------------------ consumer warps
  const int kg = warp / p.ntg, tg = warp - (warp / p.ntg) * p.ntg;
  const int g = lane >> 2, t = lane & 3;
  const int R = p.R, G = p.G;

  long long seg_start = p0;
  while (seg_start < p1) {
    int b, h, lp0, np;
    decode_page(pre, p.B, p.Hkv, seg_start, b, h, lp0, np);
    const long long seg_end = min(p1, seg_start + (np - lp0));
    const int seg = b * p.Hkv + h;
    bool bad_ctx = false;
    const int ctxb = eff_ctx(p, b, bad_ctx, FMT);
    if (FMT == 1 && bad_ctx && threadIdx.x == 0) set_err(p.dev_err, KVQ_DEVERR_POS);

    // ---- segment setup: query fragments and per-row limits
    uint32_t qf[NT][8][2];
    float qs[NT][2];
    int lim_lo[NT][2], lim_hi[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int tile = tg * NT + nt;
      const int nB = 8 * tile + g;
      float qv[32];
      if (nB < R) {
        const size_t row = ((size_t)b * p.S + nB / G) * p.Hq + h * G + nB % G;
        if (FMT == 0 || !p.q_bf16) {
          const float* qbase = FMT == 0 ? p.q_rot : static_cast<const float*>(p.q);
          const float4* src = reinterpret_cast<const float4*>(qbase + row * kD + 32 * t);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 v = src[i];
            qv[4 * i] = v.x;
            qv[4 * i + 1] = v.y;
            qv[4 * i + 2] = v.z;
            qv[4 * i + 3] = v.w;
          }
        } else {
          const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q) + row * kD + 32 * t);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint4 v = src[i];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              qv[8 * i + 2 * k] = bf16_bits_to_f32(w[k] & 0xFFFFu);
              qv[8 * i + 2 * k + 1] = bf16_bits_to_f32(w[k] >> 16);
            }
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) qv[i] = 0.0f;
      }
      float part = 0.0f;
#pragma unroll
      for (int i = 0; i < 32; ++i) part += qv[i];
      if (FMT == 0) {
        // k-step 2wi+e, slots (2t,2t+1) <- dims (8wi+2e, +4), slots (2t+8,2t+9) <- (+1, +5);
        // the second pair meets high nibbles, read as 16 c 2^-24 (unpack8_sub), so its query
        // values are divided by 16 (exact).
#pragma unroll
        for (int wi = 0; wi < 4; ++wi)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int d0 = 8 * wi + 2 * e;
            qf[nt][2 * wi + e][0] = pack_f16x2(qv[d0], qv[d0 + 4]);
            qf[nt][2 * wi + e][1] = pack_f16x2(qv[d0 + 1] * 0.0625f, qv[d0 + 5] * 0.0625f);
          }
      } else {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          qf[nt][ks][0] = pack_f16x2(qv[4 * ks], qv[4 * ks + 1]);
          qf[nt][ks][1] = pack_f16x2(qv[4 * ks + 2], qv[4 * ks + 3]);
        }
      }
      // full row sum (int4 offset term), then the sums of the rows of my accumulator columns
      part += __shfl_xor_sync(0xffffffffu, part, 1);
      part += __shfl_xor_sync(0xffffffffu, part, 2);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float tot = __shfl_sync(0xffffffffu, part, (2 * t + j) * 4);
        qs[nt][j] = tot * p.score_scale;
        const int nC = 8 * tile + 2 * t + j;
        const int r = nC < R ? nC / G : 0;
        const int hi = ctxb + r;  // last visible position
        lim_hi[nt][j] = hi;
        lim_lo[nt][j] = FMT == 0 ? 0 : max(0, hi - p.window + 1);
      }
    }

    // Softmax state per accumulator row: m = exponent base (-inf until a finite score is seen),
    // muse = the base used in the exponent (0 while m is -inf), thr = how far a score may exceed
    // the base before it is moved (scores enter the exponent as s - muse).
    float m[NT][2], muse[NT][2], thr[NT][2], l[NT][2], ov[NT][2], acc[NT][8][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        m[nt][j] = -INFINITY;
        muse[nt][j] = 0.0f;
        thr[nt][j] = -INFINITY;
        l[nt][j] = 0.0f;
        ov[nt][j] = 0.0f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[nt][i][c] = 0.0f;
    }

    // fp8 ring: the newest position written and its slot
    const int p_last = ctxb + p.S - 1;
    const int slot_last = FMT == 1 ? p_last % p.cap : 0;

    const int k_beg = (int)(seg_start - p0), k_end = (int)(seg_end - p0);
    for (int k = k_beg + ((kg - k_beg % p.nkg + p.nkg) % p.nkg); k < k_end; k += p.nkg) {
      const long long pg = p0 + k;
      const int s = k % nst;
      const int f = k / nst;
      const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[s], f & 1, p.stage_wait_ns));
      if (!ok) {
        if (lane == 0) set_err(p.dev_err, KVQ_DEVERR_TIMEOUT);
        flags[0] = 1;
      }
      if (__any_sync(0xffffffffu, flags[0] != 0)) break;
      const int lp = lp0 + (int)(pg - seg_start);
      if (valid[s]) {
        const uint8_t* st = stages + (size_t)s * kStage;
        const bool need_mask = FMT == 1 || (lp + 1) * kPage > ctxb + 1;

#pragma unroll
        for (int mt0 = 0; mt0 < 4; mt0 += MTU) {
          // ---- per-token scale/offset (int4) for the tokens of this thread's accumulator rows
          float ka[MTU][2], kb[MTU][2], va[MTU][2], vb[MTU][2];
          if (FMT == 0) {
            const uint32_t* Km = reinterpret_cast<const uint32_t*>(st + 2 * kPage * kRec4);
            const uint32_t* Vm = Km + kPage;
#pragma unroll
            for (int u = 0; u < MTU; ++u)
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                const int tok = 16 * (mt0 + u) + g + 8 * hh;
                const uint32_t mk = Km[tok], mv = Vm[tok];
                const float sk = h2f_lo(mk), ok_ = h2f_hi(mk), sv = h2f_lo(mv), ovv = h2f_hi(mv);
                ka[u][hh] = sk * p.score_scale * 16777216.0f;  // the MMA's products carry 2^-24
                kb[u][hh] = ok_;
                va[u][hh] = sv;
                vb[u][hh] = fmaf(7.5f, sv, ovv);
              }
          }

          // ---- scores
          float sc[NT][MTU][4];
          if (FMT == 0) {
            // Load every m-tile's K words first, then interleave the m-tiles' MMA chains so
            // independent accumulators hide the tensor-core latency.
            const uint8_t* Ks = st;
            uint32_t A[MTU][4], Bw[MTU][4];
#pragma unroll
            for (int u = 0; u < MTU; ++u) {
              const uint4 wa = *reinterpret_cast<const uint4*>(Ks + (16 * (mt0 + u) + g) * kRec4 + 16 * t);
              const uint4 wb = *reinterpret_cast<const uint4*>(Ks + (16 * (mt0 + u) + g + 8) * kRec4 + 16 * t);
              A[u][0] = wa.x;
              A[u][1] = wa.y;
              A[u][2] = wa.z;
              A[u][3] = wa.w;
              Bw[u][0] = wb.x;
              Bw[u][1] = wb.y;
              Bw[u][2] = wb.z;
              Bw[u][3] = wb.w;
            }
            float d[NT][MTU][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int u = 0; u < MTU; ++u)
#pragma unroll
                for (int c = 0; c < 4; ++c) d[nt][u][c] = 0.0f;
#pragma unroll
            for (int wi = 0; wi < 4; ++wi) {
              uint32_t ha[MTU][4], hb[MTU][4];
#pragma unroll
              for (int u = 0; u < MTU; ++u) {
                unpack8_sub(A[u][wi], ha[u]);
                unpack8_sub(Bw[u][wi], hb[u]);
              }
#pragma unroll
              for (int e = 0; e < 2; ++e)
#pragma unroll
                for (int u = 0; u < MTU; ++u)
#pragma unroll
                  for (int nt = 0; nt < NT; ++nt)
                    mma_16816(d[nt][u], ha[u][2 * e], hb[u][2 * e], ha[u][2 * e + 1], hb[u][2 * e + 1],
                              qf[nt][2 * wi + e][0], qf[nt][2 * wi + e][1]);
            }
#pragma unroll
            for (int u = 0; u < MTU; ++u)
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int c = 0; c < 4; ++c)
                  sc[nt][u][c] = fmaf(d[nt][u][c], ka[u][c >> 1], fmaf(kb[u][c >> 1], qs[nt][c & 1], -muse[nt][c & 1]));
          } else {
#pragma unroll
            for (int u = 0; u < MTU; ++u) {
              const int mt = mt0 + u;
              float d[NT][4];
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int c = 0; c < 4; ++c) d[nt][c] = 0.0f;
              const uint8_t* Ks = st;
              const int ta = 16 * mt + g, tb = ta + 8;  // slot & 7 == g for both tokens
              const uint4 a0 = *reinterpret_cast<const uint4*>(Ks + ta * kRec8 + 16 * ((2 * t) ^ g));
              const uint4 a1 = *reinterpret_cast<const uint4*>(Ks + ta * kRec8 + 16 * ((2 * t + 1) ^ g));
              const uint4 b0 = *reinterpret_cast<const uint4*>(Ks + tb * kRec8 + 16 * ((2 * t) ^ g));
              const uint4 b1 = *reinterpret_cast<const uint4*>(Ks + tb * kRec8 + 16 * ((2 * t + 1) ^ g));
              const uint32_t A[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
              const uint32_t Bw[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
              for (int ks = 0; ks < 8; ++ks) {
                const uint32_t x0 = e4m3x2_to_f16x2(A[ks] & 0xFFFFu), x2 = e4m3x2_to_f16x2(A[ks] >> 16);
                const uint32_t x1 = e4m3x2_to_f16x2(Bw[ks] & 0xFFFFu), x3 = e4m3x2_to_f16x2(Bw[ks] >> 16);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) mma_16816(d[nt], x0, x1, x2, x3, qf[nt][ks][0], qf[nt][ks][1]);
              }
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int c = 0; c < 4; ++c)
                  sc[nt][u][c] = fmaf(d[nt][c], p.score_scale, -muse[nt][c & 1]);
            }
          }
          if (need_mask) {
#pragma unroll
            for (int u = 0; u < MTU; ++u)
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                const int tok = 16 * (mt0 + u) + g + 8 * hh;
                int pos;
                if (FMT == 0) {
                  pos = lp * kPage + tok;
                } else {
                  const int slot = lp * kPage + tok;
                  int back = slot_last - slot;
                  if (back < 0) back += p.cap;
                  pos = p_last - back;
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                  for (int j = 0; j < 2; ++j)
                    if (pos < lim_lo[nt][j] || pos > lim_hi[nt][j]) sc[nt][u][2 * hh + j] = -INFINITY;
              }
          }

          // ---- online softmax update
          // Lazy base: scores are already relative to muse. The base moves (to the running
          // maximum, rescaling l, ov and acc) only when some score of the page exceeds it by
          // more than 8, so P stays <= 2^8 and most pages skip the cross-lane maximum. P s_V
          // enters the PV product in f16, which stays finite for P <= 2^8 while s_V < 255; a page
          // holding a larger V scale moves the base as soon as any score exceeds it, so that
          // there P <= 1 and P s_V <= 65504.
          {
            float mx[NT][2];
            bool need = false;
            bool big = false;
            if (FMT == 0) {
              float vmax = 0.0f;
#pragma unroll
              for (int u = 0; u < MTU; ++u) vmax = fmaxf(vmax, fmaxf(va[u][0], va[u][1]));
              big = vmax >= 255.0f;
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                float v = -INFINITY;
#pragma unroll
                for (int u = 0; u < MTU; ++u) v = fmaxf(v, fmaxf(sc[nt][u][j], sc[nt][u][2 + j]));
                mx[nt][j] = v;
                need |= v > (big ? fminf(thr[nt][j], 0.0f) : thr[nt][j]);
              }
            if (__any_sync(0xffffffffu, need)) {
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                  const float mt = warp_max_g(mx[nt][j]);
                  const float mnew = fmaxf(m[nt][j], muse[nt][j] + mt);
                  if (mnew != m[nt][j]) {
                    const float mu2 = mnew == -INFINITY ? 0.0f : mnew;
                    const float alpha = fast_exp2(m[nt][j] - mu2);
                    const float delta = muse[nt][j] - mu2;
                    l[nt][j] *= alpha;
                    ov[nt][j] *= alpha;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                      acc[nt][i][j] *= alpha;
                      acc[nt][i][2 + j] *= alpha;
                    }
#pragma unroll
                    for (int u = 0; u < MTU; ++u) {
                      sc[nt][u][j] += delta;
                      sc[nt][u][2 + j] += delta;
                    }
                    m[nt][j] = mnew;
                    muse[nt][j] = mu2;
                    thr[nt][j] = mnew == -INFINITY ? -INFINITY : 8.0f;
                  }
                }
            }
          }

          // ---- P and PV
#pragma unroll
          for (int u = 0; u < MTU; ++u) {
            const int mt = mt0 + u;
            uint32_t pb[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              float pr[4];
#pragma unroll
              for (int c = 0; c < 4; ++c) pr[c] = fast_exp2(sc[nt][u][c]);
              l[nt][0] += pr[0] + pr[2];
              l[nt][1] += pr[1] + pr[3];
              if (FMT == 0) {
                ov[nt][0] = fmaf(pr[0], vb[u][0], fmaf(pr[2], vb[u][1], ov[nt][0]));
                ov[nt][1] = fmaf(pr[1], vb[u][0], fmaf(pr[3], vb[u][1], ov[nt][1]));
                pb[nt][0] = movmatrix_trans(pack_f16x2_sat(pr[0] * va[u][0], pr[1] * va[u][0]));
                pb[nt][1] = movmatrix_trans(pack_f16x2_sat(pr[2] * va[u][1], pr[3] * va[u][1]));
              } else {
                pb[nt][0] = movmatrix_trans(pack_f16x2(pr[0], pr[1]));
                pb[nt][1] = movmatrix_trans(pack_f16x2(pr[2], pr[3]));
              }
            }
            const uint8_t* Vs = st + kPage * (FMT == 0 ? kRec4 : kRec8);
            const int qi = lane >> 3, r8 = lane & 7;
            if (FMT == 0) {
#pragma unroll
              for (int cc = 0; cc < 2; ++cc) {
                const int cprime = 2 * cc + (qi >> 1), th = qi & 1;
                const int tok = 16 * mt + 8 * th + r8;
                uint32_t rr[4];
                ldsm_x4_trans(rr, smem_addr(Vs + tok * kRec4 + 16 * (cprime ^ (r8 >> 1))));
#pragma unroll
                for (int ci = 0; ci < 2; ++ci) {
                  uint32_t h0[4], h1[4];
                  unpack8_v(rr[2 * ci], h0);
                  unpack8_v(rr[2 * ci + 1], h1);
#pragma unroll
                  for (int e1 = 0; e1 < 2; ++e1) {
                    const int mtd = 2 * (2 * cc + ci) + e1;
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                      mma_16816(acc[nt][mtd], h0[2 * e1], h0[2 * e1 + 1], h1[2 * e1], h1[2 * e1 + 1], pb[nt][0],
                                pb[nt][1]);
                  }
                }
              }
            } else {
#pragma unroll
              for (int cc = 0; cc < 4; ++cc) {
                const int cprime = 2 * cc + (qi >> 1), th = qi & 1;
                const int tok = 16 * mt + 8 * th + r8;
                uint32_t rr[4];
                ldsm_x4_trans(rr, smem_addr(Vs + tok * kRec8 + 16 * (cprime ^ r8)));
#pragma unroll
                for (int ci = 0; ci < 2; ++ci) {
                  const uint32_t y0 = prmt(rr[2 * ci], 0u, 0x3120u);
                  const uint32_t y1 = prmt(rr[2 * ci + 1], 0u, 0x3120u);
                  const uint32_t a0 = e4m3x2_to_f16x2(y0 & 0xFFFFu), a1 = e4m3x2_to_f16x2(y0 >> 16);
                  const uint32_t a2 = e4m3x2_to_f16x2(y1 & 0xFFFFu), a3 = e4m3x2_to_f16x2(y1 >> 16);
                  const int mtd = 2 * cc + ci;
#pragma unroll
                  for (int nt = 0; nt < NT; ++nt) mma_16816(acc[nt][mtd], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
                }
              }
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }

    // ---- segment end: the token groups' states are merged pairwise, lane by lane (every token
    // group of a tile group holds the same rows and dims in the same fragment positions), from
    // the last token group down to group 0 through one shared slot per tile group; group 0 then
    // reduces l and the offset term over its lanes and writes the CTA partial.
    float* mslot = red + (size_t)tg * NT * kMergeFloats * 32;
    for (int kk = p.nkg - 1; kk >= 1; --kk) {
      if (kg == kk) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float* q = mslot + (size_t)nt * kMergeFloats * 32 + lane;
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            q[32 * j] = m[nt][j];
            q[32 * (2 + j)] = l[nt][j];
            q[32 * (4 + j)] = ov[nt][j];
          }
#pragma unroll
          for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int c = 0; c < 4; ++c) q[32 * (6 + 4 * i + c)] = acc[nt][i][c];
        }
      }
      named_barrier(1, nwc * 32);
      if (kg == kk - 1) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const float* q = mslot + (size_t)nt * kMergeFloats * 32 + lane;
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const float mo = q[32 * j];
            const float mn = fmaxf(m[nt][j], mo);
            const float mu = mn == -INFINITY ? 0.0f : mn;
            const float a = fast_exp2(m[nt][j] - mu), bo = fast_exp2(mo - mu);
            l[nt][j] = fmaf(l[nt][j], a, q[32 * (2 + j)] * bo);
            ov[nt][j] = fmaf(ov[nt][j], a, q[32 * (4 + j)] * bo);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              acc[nt][i][j] = fmaf(acc[nt][i][j], a, q[32 * (6 + 4 * i + j)] * bo);
              acc[nt][i][2 + j] = fmaf(acc[nt][i][2 + j], a, q[32 * (6 + 4 * i + 2 + j)] * bo);
            }
            m[nt][j] = mn;
          }
        }
      }
      named_barrier(1, nwc * 32);
    }
    if (kg == 0) {
      float* dstp = p.partials + ((size_t)(blockIdx.x + seg) * R) * kPartialStride;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int tile = tg * NT + nt;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float lt = warp_sum_g(l[nt][j]);
          const float ot = warp_sum_g(ov[nt][j]);
          const int row = 8 * tile + 2 * t + j;
          if (row >= R) continue;
          float* dst = dstp + (size_t)row * kPartialStride;
          if (g == 0) {
            dst[0] = m[nt][j];
            dst[1] = lt;
          }
          const float vs = FMT == 0 ? 1.0f : p.v_scale;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int dlo = out_dim<FMT>(i, g), dhi = out_dim<FMT>(i, g + 8);
            if (FMT == 0) {  // V entered as unpack8_v values: dims of class 2 (i & 1) and 2 (i & 1) + 1
              dst[2 + dlo] = fmaf(acc[nt][i][j], v_unscale(2 * (i & 1)), ot);
              dst[2 + dhi] = fmaf(acc[nt][i][2 + j], v_unscale(2 * (i & 1) + 1), ot);
            } else {
              dst[2 + dlo] = (acc[nt][i][j] + ot) * vs;
              dst[2 + dhi] = (acc[nt][i][2 + j] + ot) * vs;
            }
          }
        }
      }
    }
    seg_start = seg_end;
  }

}

template <int FMT>
__global__ void __launch_bounds__(128) combine_kernel(const AttnParams p) {
  extern __shared__ __align__(16) int cpre[];
  volatile int* flags = cpre + p.B + 1;
  // The previous grid is the same call's attention kernel. It triggers this launch only after
  // its own wait, so every grid before it has completed, and it writes nothing but the partials
  // and the error word: the context lengths (read at L2, see eff_ctx) are taken before waiting.
  build_prefix(p, FMT, cpre, flags);
  griddep_wait();
  griddep_launch_dependents();
  __syncthreads();
  const int R = p.R;
  const int seg = blockIdx.x / R, row = blockIdx.x - (blockIdx.x / R) * R;
  const int b = seg / p.Hkv, h = seg - (seg / p.Hkv) * p.Hkv;
  const long long P = (long long)p.Hkv * cpre[p.B];
  const int n_eff = (int)min((long long)p.n_cta, P);
  const int np = cpre[b + 1] - cpre[b];
  const long long first_pg = (long long)p.Hkv * cpre[b] + (long long)h * np;
  const int c0 = (int)cta_of(first_pg, P, n_eff), c1 = (int)cta_of(first_pg + np - 1, P, n_eff);
  const int d = threadIdx.x;
  // chunks of up to 8 partials: all loads of a chunk are issued before any is used; the chunk
  // is merged with log-sum-exp weights against its own maximum, then folded into the total
  float M = -INFINITY, lsum = 0.0f, a = 0.0f;
  for (int cb = c0; cb <= c1; cb += 8) {
    float mv[8], lv[8], av[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (cb + k <= c1) {
        const float* src = p.partials + ((size_t)(cb + k + seg) * R + row) * kPartialStride;
        mv[k] = src[0];
        lv[k] = src[1];
        av[k] = src[2 + d];
      } else {
        mv[k] = -INFINITY;
        lv[k] = 0.0f;
        av[k] = 0.0f;
      }
    }
    float Mc = mv[0];
#pragma unroll
    for (int k = 1; k < 8; ++k) Mc = fmaxf(Mc, mv[k]);
    if (Mc == -INFINITY) continue;  // nothing visible in this chunk
    float lc = 0.0f, ac = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float w = fast_exp2(mv[k] - Mc);
      lc += w * lv[k];
      ac += w * av[k];
    }
    if (M == -INFINITY) {
      M = Mc;
      lsum = lc;
      a = ac;
    } else {
      const float Mn = fmaxf(M, Mc);
      const float so = fast_exp2(M - Mn), sc = fast_exp2(Mc - Mn);
      lsum = lsum * so + lc * sc;
      a = a * so + ac * sc;
      M = Mn;
    }
  }
  const int r = row / p.G, gi = row - (row / p.G) * p.G;
  p.out[(((size_t)b * p.S + r) * p.Hq + h * p.G + gi) * kD + d] = a / lsum;
}

struct DevCache {
  int sm = 0;
  bool attr[2][4] = {{false}};
  size_t occ_smem[2][4] = {{0}};  // occupancy cache: last (smem, threads) queried per instantiation
  int occ_threads[2][4] = {{0}};
  int occ[2][4] = {{0}};
};
DevCache g_dev[64];
std::mutex g_dev_mu;  // guards g_dev (launch-configuration caches shared by host threads)

template <int FMT, int NT>
cudaError_t launch_attn_t(AttnParams& p, size_t smem, int threads, long long p_max, cudaStream_t stream) {
  int dev = 0;
  cudaGetDevice(&dev);
  cudaError_t e = cudaSuccess;
  int occ = 1, sm = 1;
  {
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DevCache& dc = g_dev[(dev >= 0 && dev < 64) ? dev : 0];
    if (dc.sm == 0) {
      int n = 0;
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
      dc.sm = n > 0 ? n : 1;
    }
    if (!dc.attr[FMT][NT]) {
      e = cudaFuncSetAttribute(attn_kernel<FMT, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, 220 * 1024);
      if (e != cudaSuccess) return e;
      dc.attr[FMT][NT] = true;
    }
    if (dc.occ_smem[FMT][NT] != smem || dc.occ_threads[FMT][NT] != threads) {
      int o = 0;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, attn_kernel<FMT, NT>, threads, smem);
      if (e != cudaSuccess) return e;
      dc.occ[FMT][NT] = std::max(o, 1);
      dc.occ_smem[FMT][NT] = smem;
      dc.occ_threads[FMT][NT] = threads;
    }
    occ = dc.occ[FMT][NT];
    sm = dc.sm;
  }
  long long grid = std::min<long long>((long long)sm * occ, kMaxCtas);
  grid = std::max<long long>(1, std::min(grid, p_max));
  p.n_cta = (int)grid;
  // both grids may start while the previous one on the stream finishes (each waits for it
  // before reading anything)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3((unsigned)threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, attn_kernel<FMT, NT>, p);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3((unsigned)(p.B * p.Hkv * p.R), 1, 1);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = (p.B + 1 + 4) * sizeof(int);
  return cudaLaunchKernelEx(&cfg, combine_kernel<FMT>, p);
}

}  // namespace

std::atomic<unsigned long long> g_stage_wait_ns{kWaitLimitNs};

void set_stage_wait_limit_ns(unsigned long long ns) { g_stage_wait_ns.store(ns, std::memory_order_relaxed); }

size_t workspace_qrot_bytes(int B, int S, int Hq) { return align_up((size_t)B * S * Hq * kD * 4, 256); }

size_t workspace_partials_bytes(int B, int S, int Hq, int Hkv) {
  const int G = Hq / Hkv;
  return align_up(((size_t)kMaxCtas + (size_t)B * Hkv) * S * G * kPartialStride * 4, 256);
}

cudaError_t launch_attention(const AttnJob& job, cudaStream_t stream) {
  AttnParams p{};
  p.stage_wait_ns = g_stage_wait_ns.load(std::memory_order_relaxed);
  p.B = job.B;
  p.S = job.S;
  p.Hq = job.Hq;
  p.Hkv = job.Hkv;
  p.G = job.Hq / job.Hkv;
  p.R = p.S * p.G;
  p.ctx = job.ctx;
  p.out = job.out;
  p.partials = job.partials;
  p.dev_err = job.dev_err;
  long long p_max;
  if (job.fmt == 0) {
    p.blocks = job.cache.pages;
    p.block_table = job.cache.block_table;
    p.max_pages = job.cache.max_pages_per_seq;
    p.num_pages = job.cache.num_pages;
    p.q_rot = job.q_rot;
    p.score_scale = job.sm_scale * kLog2e;
    p_max = (long long)p.Hkv * p.B * p.max_pages;
  } else {
    p.blocks = job.ring.data;
    p.cap = job.ring.capacity;
    p.window = job.window;
    p.v_scale = job.v_scale;
    p.q = job.q;
    p.q_bf16 = job.q_bf16;
    p.score_scale = job.sm_scale * kLog2e * job.k_scale;
    p_max = (long long)p.Hkv * p.B * (p.cap / kPage);
  }
  const int ntiles = (p.R + 7) / 8;
  int NT;
  if (ntiles <= 3) {
    NT = ntiles;
    p.ntg = 1;
    p.nkg = NT == 1 ? KVQ_TOKEN_GROUPS : (job.fmt == 0 ? KVQ_TILES3_TOKEN_GROUPS : 4);
    p.nstages = NT == 1 ? KVQ_STAGES_INT4 : (job.fmt == 0 ? KVQ_TILES3_STAGES : 8);
  } else {
    NT = (ntiles + 1) / 2;
    p.ntg = 2;
    p.nkg = job.fmt == 0 ? KVQ_TILES6_TOKEN_GROUPS : 2;
    p.nstages = job.fmt == 0 ? KVQ_TILES6_STAGES : 4;
  }
  if (job.fmt == 1) {  // window rings too large for one cluster per (sequence, KV head)
    p.nkg = NT == 1 ? 4 : 2;
    p.nstages = 4;
  }
  p.rows_pad = p.ntg * NT * 8;
  if (p.nstages % p.nkg != 0) return cudaErrorInvalidConfiguration;  // see the static_assert above
  const int threads = (p.ntg * p.nkg + 1) * 32;
  const SmemLayout L(job.fmt, p.nstages, p.B, p.nkg, p.rows_pad);
  const size_t smem = L.total;
  if (job.fmt == 0) {
    switch (NT) {
      case 1: return launch_attn_t<0, 1>(p, smem, threads, p_max, stream);
      case 2: return launch_attn_t<0, 2>(p, smem, threads, p_max, stream);
      default: return launch_attn_t<0, 3>(p, smem, threads, p_max, stream);
    }
  }
  switch (NT) {
    case 1: return launch_attn_t<1, 1>(p, smem, threads, p_max, stream);
    case 2: return launch_attn_t<1, 2>(p, smem, threads, p_max, stream);
    default: return launch_attn_t<1, 3>(p, smem, threads, p_max, stream);
  }
}

}  // namespace kvq
