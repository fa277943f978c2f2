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
//        read as f16 1024 + c (low nibbles) or 1024 + 16c (high nibbles, whose query values
//        are divided by 16), B = 16 dims x 8 query rows of q~ in f16; the accumulator starts at
//        -1024 sum(q~ fragment), so it holds sum q~ c exactly up to fp32 rounding;
//   score = log2(e)*sm_scale*(s_K*dot + o_K*sum(q~)) -- scale and offset per token;
//   online softmax with exp2 against a lazily moved base (moved only when a score passes it
//        by more than 8, or by anything on pages with a V scale of 255 or more);
//   PV on tensor cores: A = 16 dims x 16 tokens of V codes read as f16 subnormals
//        (c - 7.5) 2^(k - 23), B = 16 tokens x 8 rows of p*s_V in f16 (movmatrix transposes
//        the QK accumulator), plus
//        sum_j p_j (o_V + 7.5 s_V) added per row; the partial undoes 2^(k - 23) per dim.

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
// K codes enter QK^T as 1024+c (no per-element bias subtraction); see unpack8_biased.
#ifndef KVQ_K_BIASED
#define KVQ_K_BIASED 1
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
    float negbias[NT][2];  // biased K path: -1024 * sum of the row's query fragment values
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
        // the second pair meets high nibbles, read as 16*code in the biased K path, so its
        // query values are divided by 16 (exact).
        const float hs = KVQ_K_BIASED ? 0.0625f : 1.0f;
        float bsum = 0.0f;
#pragma unroll
        for (int wi = 0; wi < 4; ++wi)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int d0 = 8 * wi + 2 * e;
            const uint32_t b0 = pack_f16x2(qv[d0], qv[d0 + 4]);
            const uint32_t b1 = pack_f16x2(qv[d0 + 1] * hs, qv[d0 + 5] * hs);
            qf[nt][2 * wi + e][0] = b0;
            qf[nt][2 * wi + e][1] = b1;
            bsum += (h2f_lo(b0) + h2f_hi(b0)) + (h2f_lo(b1) + h2f_hi(b1));
          }
        bsum += __shfl_xor_sync(0xffffffffu, bsum, 1);
        bsum += __shfl_xor_sync(0xffffffffu, bsum, 2);
#pragma unroll
        for (int j = 0; j < 2; ++j)
          negbias[nt][j] = KVQ_K_BIASED ? -1024.0f * __shfl_sync(0xffffffffu, bsum, (2 * t + j) * 4) : 0.0f;
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
                ka[u][hh] = sk * p.score_scale;
                kb[u][hh] = KVQ_K_BIASED ? ok_ : fmaf(8.0f, sk, ok_);
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
                for (int c = 0; c < 4; ++c) d[nt][u][c] = negbias[nt][c & 1];
#pragma unroll
            for (int wi = 0; wi < 4; ++wi) {
              uint32_t ha[MTU][4], hb[MTU][4];
#pragma unroll
              for (int u = 0; u < MTU; ++u) {
                if (KVQ_K_BIASED) {
                  unpack8_biased(A[u][wi], ha[u]);
                  unpack8_biased(Bw[u][wi], hb[u]);
                } else {
                  unpack8_centred(A[u][wi], ha[u]);
                  unpack8_centred(Bw[u][wi], hb[u]);
                }
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

// ------------------------------------------------------------ many query rows per KV head
// For S x G > 8 query rows (verify blocks) the rows span several 8-row tiles. Converting each
// page's 4-bit codes once per tile would repeat the dominant ALU work, so here the conversion
// is done once per page into shared f16 tiles that every tile warp reads with ldmatrix:
//
//   warp 0          producer: page-head blocks into kVStages int4 stages (produce_pages)
//   kConvWarps      converters: K codes -> f16 biased (1024 + c / 1024 + 16c, see
//                   unpack8_biased), V codes -> f16 subnormals (c - 7.5) 2^(k - 23) (see
//                   unpack8_v), per-token scale/offset -> fp32, into one of kVBufs tile
//                   buffers; each converts an equal share of the 64 tokens
//   T tile warps    one per 8 query rows: QK^T, online softmax and PV on tensor
//                   cores over every page of the CTA's range, partial per segment and row
//
// A tile buffer holds K16 [64 tokens][16 chunks of 16 B], V16 the same, meta [64] float4. Chunk
// j of a token row holds the eight f16 values of code word j (dims 8j .. 8j+7) in the order the
// unpack produces them (dims 8j + {0,4,1,5,2,6,3,7}) and sits at chunk position j ^ (token & 7),
// so the eight rows an ldmatrix 8x8 matrix reads fall in eight different bank groups.
constexpr int kVStages = 8;
constexpr int kVBufs = 3;
constexpr int kTileRow = 256;                                // bytes per token row of an f16 tile
constexpr int kVBuf = 2 * kPage * kTileRow + kPage * 16;     // K16, V16, meta
#ifndef KVQ_VERIFY_CONV
#define KVQ_VERIFY_CONV 2
#endif
// Row tiles (8 query rows each) from which the environment variable KVQ_MANY_ROWS_KERNEL may
// select this shared-tile kernel ("tile") or the tcgen05 kernel ("tcgen05") instead of the split
// kernel, which is the default for every call (faster at 5 and 6 tiles as well: 516 against
// 560 us at S = 8, GQA 5, 64 x 16,384).
#ifndef KVQ_VERIFY_MIN_TILES
#define KVQ_VERIFY_MIN_TILES 5
#endif
constexpr int kConvWarps = KVQ_VERIFY_CONV;  // 64 / kConvWarps tokens each
static_assert(64 % (2 * kConvWarps) == 0, "converter warps split the page's tokens in pairs of rows");

struct VerifyLayout {
  size_t bufs, full, empty, ready, freeb, valid, vvalid, pre, flags, total;
  __host__ __device__ explicit VerifyLayout(int B) {
    bufs = (size_t)kVStages * kStage4;  // int4 stages first, from offset 0
    full = bufs + (size_t)kVBufs * kVBuf;
    empty = full + 8 * kVStages;
    ready = empty + 8 * kVStages;
    freeb = ready + 8 * kVBufs;
    valid = freeb + 8 * kVBufs;
    vvalid = valid + 4 * kVStages;
    pre = vvalid + 4 * kVBufs;
    flags = align_up(pre + 4 * (size_t)(B + 1), 16);
    total = flags + 16;
  }
};

// Dim held by element e (0..7) of chunk j of a tile row.
__device__ __forceinline__ int tile_dim(int j, int e) { return 8 * j + (e >> 1) + 4 * (e & 1); }

__global__ void __launch_bounds__((1 + kConvWarps + 6) * 32, 1) attn_verify_kernel(const AttnParams p) {
  constexpr int kTokPerConv = kPage / kConvWarps;
  extern __shared__ __align__(128) uint8_t smem[];
  const VerifyLayout L(p.B);
  uint8_t* stages = smem;
  uint8_t* bufs = smem + L.bufs;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.full);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.empty);
  uint64_t* ready = reinterpret_cast<uint64_t*>(smem + L.ready);
  uint64_t* freeb = reinterpret_cast<uint64_t*>(smem + L.freeb);
  volatile int* valid = reinterpret_cast<volatile int*>(smem + L.valid);
  volatile int* vvalid = reinterpret_cast<volatile int*>(smem + L.vvalid);
  int* pre = reinterpret_cast<int*>(smem + L.pre);
  volatile int* flags = reinterpret_cast<volatile int*>(smem + L.flags);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = p.ntg;  // tile warps

  griddep_wait();
  griddep_launch_dependents();
  build_prefix(p, 0, pre, flags);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConvWarps);
    }
    for (int b = 0; b < kVBufs; ++b) {
      mbar_init(&ready[b], kConvWarps);
      mbar_init(&freeb[b], T);
    }
  }
  fence_barrier_init();
  __syncthreads();

  if (blockIdx.x == 0 && threadIdx.x == 0 && flags[1]) set_err(p.dev_err, KVQ_DEVERR_POS);
  const long long P = (long long)p.Hkv * pre[p.B];
  const int n_eff = (int)min((long long)p.n_cta, P);
  if ((int)blockIdx.x >= n_eff) return;
  const long long p0 = (long long)blockIdx.x * P / n_eff;
  const long long p1 = (long long)(blockIdx.x + 1) * P / n_eff;
  const int npages = (int)(p1 - p0);

  if (warp == 0) {
    produce_pages<0>(p, pre, stages, full, empty, valid, flags, kVStages, p0, p1, lane);
    return;
  }

  // ------------------------------------------------------------ converter warps
  if (warp <= kConvWarps) {
    const int cw = warp - 1;
    for (int k = 0; k < npages; ++k) {
      const int s = k % kVStages, b = k % kVBufs;
      bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[s], (uint32_t)(k / kVStages) & 1u));
      if (ok && k >= kVBufs)  // the buffer's previous page has been released by every tile warp
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&freeb[b], (uint32_t)(k / kVBufs - 1) & 1u));
      if (!ok) {
        if (lane == 0) set_err(p.dev_err, KVQ_DEVERR_TIMEOUT);
        flags[0] = 1;
        break;
      }
      const uint8_t* st4 = stages + (size_t)s * kStage4;
      uint8_t* buf = bufs + (size_t)b * kVBuf;
      const int vpage = valid[s];
      if (cw == 0 && lane == 0) vvalid[b] = vpage;
      if (vpage) {
        // lane = (row of a token pair, code word j); all loads of the share are issued first
        constexpr int kIt = kTokPerConv / 2;
        const int j = lane & 15;
        uint32_t kw[kIt], vw[kIt];
#pragma unroll
        for (int it = 0; it < kIt; ++it) {
          const int tok = kTokPerConv * cw + 2 * it + (lane >> 4);
          kw[it] = *reinterpret_cast<const uint32_t*>(st4 + tok * kRec4 + 4 * j);
          // V records: 16-byte chunk c of slot s stored at chunk c ^ ((s >> 1) & 3)
          vw[it] = *reinterpret_cast<const uint32_t*>(st4 + kPage * kRec4 + tok * kRec4 +
                                                      16 * ((j >> 2) ^ ((tok >> 1) & 3)) + 4 * (j & 3));
        }
#pragma unroll
        for (int it = 0; it < kIt; ++it) {
          const int tok = kTokPerConv * cw + 2 * it + (lane >> 4);
          uint32_t h[4];
          unpack8_biased(kw[it], h);
          *reinterpret_cast<uint4*>(buf + tok * kTileRow + 16 * (j ^ (tok & 7))) = make_uint4(h[0], h[1], h[2], h[3]);
          unpack8_v(vw[it], h);
          *reinterpret_cast<uint4*>(buf + kPage * kTileRow + tok * kTileRow + 16 * (j ^ (tok & 7))) =
              make_uint4(h[0], h[1], h[2], h[3]);
        }
        if (lane < kTokPerConv) {
          const int tok = kTokPerConv * cw + lane;
          const uint32_t* meta = reinterpret_cast<const uint32_t*>(st4 + 2 * kPage * kRec4);
          const uint32_t mk = meta[tok], mv = meta[kPage + tok];
          const float sv = h2f_lo(mv);
          reinterpret_cast<float4*>(buf + 2 * kPage * kTileRow)[tok] =
              make_float4(h2f_lo(mk) * p.score_scale, h2f_hi(mk), sv, fmaf(7.5f, sv, h2f_hi(mv)));
        }
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&ready[b]);
        mbar_arrive(&empty[s]);
      }
    }
    return;
  }

  // ------------------------------------------------------------ tile warps
  const int tg = warp - 1 - kConvWarps;
  const int g = lane >> 2, t = lane & 3;
  const int R = p.R, G = p.G;
  long long seg_start = p0;
  int k = 0;  // page index within the CTA's range
  while (seg_start < p1) {
    int b, h, lp0, np;
    decode_page(pre, p.B, p.Hkv, seg_start, b, h, lp0, np);
    const long long seg_end = min(p1, seg_start + (np - lp0));
    const int seg = b * p.Hkv + h;
    bool bad_ctx = false;
    const int ctxb = eff_ctx(p, b, bad_ctx, 0);

    // ---- query fragments of this warp's 8 rows. Element pairs of k-step ks: b0 <- dims
    // (16 ks + t, 16 ks + t + 4), b1 <- (16 ks + 8 + t, 16 ks + 12 + t) (the tile's dim order);
    // odd t meets high nibbles (1024 + 16c), so those query values are divided by 16 (exact).
    uint32_t qf[8][2];
    float qs[2], negbias[2];
    int lim_hi[2];
    {
      const int nB = 8 * tg + g;
      float qv[32];  // qv[4 ks + i] = q~[dim 16 ks + t + 4 i]
      if (nB < R) {
        const float* qrow = p.q_rot + (((size_t)b * p.S + nB / G) * p.Hq + h * G + nB % G) * kD;
#pragma unroll
        for (int m = 0; m < 32; ++m) qv[m] = qrow[4 * m + t];
      } else {
#pragma unroll
        for (int m = 0; m < 32; ++m) qv[m] = 0.0f;
      }
      float part = 0.0f, bsum = 0.0f;
      const float hs = (t & 1) ? 0.0625f : 1.0f;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t b0 = pack_f16x2(qv[4 * ks] * hs, qv[4 * ks + 1] * hs);
        const uint32_t b1 = pack_f16x2(qv[4 * ks + 2] * hs, qv[4 * ks + 3] * hs);
        qf[ks][0] = b0;
        qf[ks][1] = b1;
        bsum += (h2f_lo(b0) + h2f_hi(b0)) + (h2f_lo(b1) + h2f_hi(b1));
#pragma unroll
        for (int i = 0; i < 4; ++i) part += qv[4 * ks + i];
      }
      part += __shfl_xor_sync(0xffffffffu, part, 1);
      part += __shfl_xor_sync(0xffffffffu, part, 2);
      bsum += __shfl_xor_sync(0xffffffffu, bsum, 1);
      bsum += __shfl_xor_sync(0xffffffffu, bsum, 2);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        qs[j] = __shfl_sync(0xffffffffu, part, (2 * t + j) * 4) * p.score_scale;
        negbias[j] = -1024.0f * __shfl_sync(0xffffffffu, bsum, (2 * t + j) * 4);
        const int nC = 8 * tg + 2 * t + j;
        lim_hi[j] = ctxb + (nC < R ? nC / G : 0);
      }
    }

    // lazy exponent base, as in attn_kernel: m, muse, thr per accumulator row
    float m[2] = {-INFINITY, -INFINITY}, muse[2] = {0.0f, 0.0f}, thr[2] = {-INFINITY, -INFINITY};
    float l[2] = {0.0f, 0.0f}, ov[2] = {0.0f, 0.0f}, acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[i][c] = 0.0f;

    for (long long pg = seg_start; pg < seg_end; ++pg, ++k) {
      const int bi = k % kVBufs;
      const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&ready[bi], (uint32_t)(k / kVBufs) & 1u));
      if (!ok) {
        if (lane == 0) set_err(p.dev_err, KVQ_DEVERR_TIMEOUT);
        flags[0] = 1;
      }
      if (__any_sync(0xffffffffu, flags[0] != 0)) break;
      const int lp = lp0 + (int)(pg - seg_start);
      if (vvalid[bi]) {
        const uint8_t* buf = bufs + (size_t)bi * kVBuf;
        const uint32_t Kt = smem_addr(buf), Vt = smem_addr(buf + kPage * kTileRow);
        const float4* meta = reinterpret_cast<const float4*>(buf + 2 * kPage * kTileRow);
        const bool need_mask = (lp + 1) * kPage > ctxb + 1;

        // ---- scores for the page's 4 m-tiles (16 tokens each), chains interleaved over m-tiles
        float d[4][4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int c = 0; c < 4; ++c) d[u][c] = negbias[c & 1];
        const int arow = (lane & 7) + 8 * ((lane >> 3) & 1), achunk = lane >> 4;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          uint32_t a[4][4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int tok = 16 * u + arow, ch = 2 * ks + achunk;
            ldsm_x4(a[u], Kt + tok * kTileRow + 16 * (ch ^ (tok & 7)));
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) mma_16816(d[u], a[u][0], a[u][1], a[u][2], a[u][3], qf[ks][0], qf[ks][1]);
        }
        float sc[4][4], va[4][2], vb[4][2];
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const float4 mt = meta[16 * u + g + 8 * hh];
            va[u][hh] = mt.z;
            vb[u][hh] = mt.w;
#pragma unroll
            for (int j = 0; j < 2; ++j) sc[u][2 * hh + j] = fmaf(d[u][2 * hh + j], mt.x, fmaf(mt.y, qs[j], -muse[j]));
          }
        if (need_mask) {
#pragma unroll
          for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const int pos = lp * kPage + 16 * u + g + 8 * hh;
#pragma unroll
              for (int j = 0; j < 2; ++j)
                if (pos > lim_hi[j]) sc[u][2 * hh + j] = -INFINITY;
            }
        }

        // ---- online softmax (lazy base: moved only when a score exceeds it by more than 8,
        // or by anything on a page holding a V scale >= 255; see attn_kernel)
        {
          float mx[2];
          bool need = false;
          float vmax = 0.0f;
#pragma unroll
          for (int u = 0; u < 4; ++u) vmax = fmaxf(vmax, fmaxf(va[u][0], va[u][1]));
          const bool big = vmax >= 255.0f;
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            float v = -INFINITY;
#pragma unroll
            for (int u = 0; u < 4; ++u) v = fmaxf(v, fmaxf(sc[u][j], sc[u][2 + j]));
            mx[j] = v;
            need |= v > (big ? fminf(thr[j], 0.0f) : thr[j]);
          }
          if (__any_sync(0xffffffffu, need)) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const float mnew = fmaxf(m[j], muse[j] + warp_max_g(mx[j]));
              if (mnew != m[j]) {
                const float mu2 = mnew == -INFINITY ? 0.0f : mnew;
                const float alpha = fast_exp2(m[j] - mu2);
                const float delta = muse[j] - mu2;
                l[j] *= alpha;
                ov[j] *= alpha;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  acc[i][j] *= alpha;
                  acc[i][2 + j] *= alpha;
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  sc[u][j] += delta;
                  sc[u][2 + j] += delta;
                }
                m[j] = mnew;
                muse[j] = mu2;
                thr[j] = mnew == -INFINITY ? -INFINITY : 8.0f;
              }
            }
          }
        }

        // ---- P and PV (A = V^T from the f16 V tile with ldmatrix.trans)
        const int vtok = (lane & 7) + 8 * (lane >> 4), vchunk = (lane >> 3) & 1;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float pr[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) pr[c] = fast_exp2(sc[u][c]);
          l[0] += pr[0] + pr[2];
          l[1] += pr[1] + pr[3];
          ov[0] = fmaf(pr[0], vb[u][0], fmaf(pr[2], vb[u][1], ov[0]));
          ov[1] = fmaf(pr[1], vb[u][0], fmaf(pr[3], vb[u][1], ov[1]));
          const uint32_t pb0 = movmatrix_trans(pack_f16x2_sat(pr[0] * va[u][0], pr[1] * va[u][0]));
          const uint32_t pb1 = movmatrix_trans(pack_f16x2_sat(pr[2] * va[u][1], pr[3] * va[u][1]));
          const int tok = 16 * u + vtok;
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) {
            const int ch = 2 * cc + vchunk;
            uint32_t a[4];
            ldsm_x4_trans(a, Vt + tok * kTileRow + 16 * (ch ^ (tok & 7)));
            mma_16816(acc[cc], a[0], a[1], a[2], a[3], pb0, pb1);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&freeb[bi]);
    }

    // ---- segment end: this warp's rows of the CTA partial
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float lt = warp_sum_g(l[j]);
      const float ot = warp_sum_g(ov[j]);
      const int row = 8 * tg + 2 * t + j;
      if (row < R) {
        float* dst = p.partials + ((size_t)(blockIdx.x + seg) * R + row) * kPartialStride;
        if (g == 0) {
          dst[0] = m[j];
          dst[1] = lt;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int d0 = tile_dim(2 * i, g), d1 = tile_dim(2 * i + 1, g);
          dst[2 + d0] = fmaf(acc[i][j], v_unscale(d0 & 3), ot);  // V tiles hold unpack8_v values
          dst[2 + d1] = fmaf(acc[i][2 + j], v_unscale(d1 & 3), ot);
        }
      }
    }
    if (__any_sync(0xffffffffu, flags[0] != 0)) break;
    seg_start = seg_end;
  }
}

// ------------------------------------------------------------ many query rows: tcgen05 variant
// The shared-tile kernel above is bound by shared-memory reads: every 8-row tile warp reads the
// page's f16 tiles through ldmatrix. Here the two contractions run on the asynchronous tensor
// cores (tcgen05.mma, accumulators in tensor memory), so each tile is read once per product for
// all query rows. Work unit: up to two pages (128 tokens) of one segment.
//
//   warp 0       producer: page-head blocks into kTcStages int4 stages (produce_pages)
//   warps 1-2    converters: K codes -> K^ (unpack8_biased values), V codes -> V^ (unpack8_v
//                values), per-token fp32 (s_K * score scale, o_K, s_V, o_V + 7.5 s_V); K^ and
//                V^ token-major, 128-byte rows of 64 dims, 128-byte swizzle, dims in the
//                unpacked order 8w + {0, 4, 1, 5, 2, 6, 3, 7}
//   warp 3       MMA: S = K^ Q'^T into tensor memory (M = 128 tokens, N = rows rounded up to
//                16, K = 128 dims, K-major operands); O += V^T P (M = 128 dims, N = rows,
//                K = 128 tokens; both operands token-major, i.e. MN-major)
//   warps 4-15   softmax: thread = token (tensor-memory lane 32 (warp % 4) + lane), rows split
//                in three groups of 16 between warps w, w + 4 and w + 8; lazy exponent base as in
//                attn_kernel; P s_V written token-major (f16) for the PV product
//
// Q' is the query with the high-nibble dims divided by 16 (K^ holds 1024 + c and 1024 + 16c);
// the bias 1024 sum(Q') of each row is subtracted from S in fp32. Every wait is bounded; the
// softmax warps take every decision that steers their named barriers through barrier
// reductions, so they always meet at the same barriers.
constexpr int kTcStages = 4;
constexpr int kTcConv = 2;
constexpr int kTcSoft = 12;
constexpr int kTcThreads = (1 + kTcConv + 1 + kTcSoft) * 32;
constexpr int kTcHalf = 16;  // rows per softmax thread (three row groups)
constexpr int kTcMaxRows = 48;

struct TcLayout {  // offsets from the 1024-byte aligned start of dynamic shared memory
  size_t kt, vt, pt, qt, meta, stages, bars, valid, vvalid, flags, taddr, rowc, rowst, ovrow, rowm, red, pre, total;
  __host__ __device__ explicit TcLayout(int B) {
    kt = 0;                     // [2][2 dim-atoms][128 tokens][128 B]
    vt = kt + 2 * 32768;        // [2][2 dim-atoms][128 tokens][128 B]
    pt = vt + 2 * 32768;        // [2][128 tokens][128 B] (rows 0..63)
    qt = pt + 2 * 16384;        // [2 dim-atoms][48 rows][128 B]
    meta = qt + 2 * 6144;       // [2][128] float4
    stages = meta + 2 * 2048;   // kTcStages int4 stages
    bars = stages + (size_t)kTcStages * kStage4;
    valid = bars + 8 * 32;
    vvalid = valid + 4 * kTcStages;  // [2][2]
    flags = vvalid + 16;
    taddr = flags + 32;
    rowc = align_up(taddr + 16, 16);     // [48] float4: -bias, qs, -muse, thr
    rowst = rowc + 16 * kTcMaxRows;      // [48] m
    ovrow = rowst + 4 * kTcMaxRows;      // [48] offset sums of the finished segment
    rowm = ovrow + 4 * kTcMaxRows;       // [12][16] per-warp row maxima
    red = rowm + 4 * kTcSoft * kTcHalf;  // [12][16][2] per-warp l, ov sums
    pre = red + 8 * kTcSoft * kTcHalf;
    total = pre + 4 * (size_t)(B + 1);
  }
};

// Unit iterator shared by all roles: consecutive pairs of pages within each segment of the
// CTA's range.
struct TcUnits {
  const AttnParams& p;
  const int* pre;
  long long seg_start, seg_end, p1;
  int b, h, lp0, np, j0, kseg, sidx;
  __device__ TcUnits(const AttnParams& p_, const int* pre_, long long p0, long long p1_)
      : p(p_), pre(pre_), seg_start(p0), seg_end(p0), p1(p1_), b(0), h(0), lp0(0), np(0), j0(0), kseg(0), sidx(-1) {}
  // advance to the next unit; false at the end. first = the unit starts a segment.
  __device__ bool next(bool& first) {
    j0 += 2;
    first = false;
    if (sidx < 0 || seg_start + j0 >= seg_end) {
      if (sidx >= 0) {
        kseg += (int)(seg_end - seg_start);
        seg_start = seg_end;
      }
      if (seg_start >= p1) return false;
      decode_page(pre, p.B, p.Hkv, seg_start, b, h, lp0, np);
      seg_end = min(p1, seg_start + (np - lp0));
      j0 = 0;
      ++sidx;
      first = true;
    }
    return true;
  }
  __device__ int npg() const { return (int)min(2LL, seg_end - seg_start - j0); }
  __device__ int k0() const { return kseg + j0; }   // CTA page index of the unit's first page
  __device__ int lp() const { return lp0 + j0; }    // sequence page of the unit's first page
  __device__ bool last() const { return seg_start + j0 + 2 >= seg_end; }  // last unit of its segment
};

__device__ __forceinline__ int tc_chunk(int row, int c) { return row * 128 + ((c ^ (row & 7)) << 4); }
__device__ __forceinline__ int tc_dim(int m) {  // dim at position m of a unpacked 8-dim group
  return 8 * (m >> 3) + ((m & 1) ? 4 : 0) + ((m & 7) >> 1);
}

__global__ void __launch_bounds__(kTcThreads, 1) attn_tc_kernel(const AttnParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const TcLayout L(p.B);
  uint8_t* stages = smem + L.stages;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  // Buffers of unit u: K^, V^, meta, S (tensor memory) and P, all u % 2.
  uint64_t* full = bars;             // [4]
  uint64_t* empty = bars + 4;        // [4]
  uint64_t* tready = bars + 8;       // [2] unit converted -> MMA / softmax
  uint64_t* tfree = bars + 10;       // [2] PV(u) done -> buffers free
  uint64_t* sfull = bars + 12;       // [2] QK(u) done
  uint64_t* sfree = bars + 14;       // [2] S of unit u read
  uint64_t* pready = bars + 16;      // [2] P of unit u written
  uint64_t* qready = bars + 18;      // Q' of the next segment written
  uint64_t* ofree = bars + 19;       // O of the finished segment read
  uint64_t* fin = bars + 20;         // final MMA completion
  volatile int* valid = reinterpret_cast<volatile int*>(smem + L.valid);
  volatile int* vvalid = reinterpret_cast<volatile int*>(smem + L.vvalid);
  volatile int* flags = reinterpret_cast<volatile int*>(smem + L.flags);
  uint32_t* taddr_s = reinterpret_cast<uint32_t*>(smem + L.taddr);
  float4* rowc = reinterpret_cast<float4*>(smem + L.rowc);
  float* rowst = reinterpret_cast<float*>(smem + L.rowst);
  float* ovrow = reinterpret_cast<float*>(smem + L.ovrow);
  float* rowm = reinterpret_cast<float*>(smem + L.rowm);
  float* red = reinterpret_cast<float*>(smem + L.red);
  int* pre = reinterpret_cast<int*>(smem + L.pre);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  griddep_wait();
  griddep_launch_dependents();
  build_prefix(p, 0, pre, flags);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kTcConv);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tready[b], kTcConv);
      mbar_init(&tfree[b], 1);
      mbar_init(&sfull[b], 1);
      mbar_init(&sfree[b], kTcSoft);
      mbar_init(&pready[b], kTcSoft);
    }
    mbar_init(qready, 1);
    mbar_init(ofree, 1);
    mbar_init(fin, 1);
  }
  // V^ tiles start finite (a one-page unit multiplies the other page's rows by P = 0)
  for (int i = threadIdx.x; i < 2 * 32768 / 16; i += kTcThreads)
    reinterpret_cast<uint4*>(smem + L.vt)[i] = make_uint4(0u, 0u, 0u, 0u);
  for (int i = threadIdx.x; i < 2 * 16384 / 16; i += kTcThreads)
    reinterpret_cast<uint4*>(smem + L.pt)[i] = make_uint4(0u, 0u, 0u, 0u);
  for (int i = threadIdx.x; i < 2 * 6144 / 16; i += kTcThreads)
    reinterpret_cast<uint4*>(smem + L.qt)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_barrier_init();
  fence_proxy_async_shared();
  if (warp == 3) tmem_alloc_256(taddr_s);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *taddr_s;

  if (blockIdx.x == 0 && threadIdx.x == 0 && flags[1]) set_err(p.dev_err, KVQ_DEVERR_POS);
  const long long P = (long long)p.Hkv * pre[p.B];
  const int n_eff = (int)min((long long)p.n_cta, P);
  const bool active = (int)blockIdx.x < n_eff;
  const long long p0 = active ? (long long)blockIdx.x * P / n_eff : 0;
  const long long p1 = active ? (long long)(blockIdx.x + 1) * P / n_eff : 0;
  const int R = p.R, G = p.G;
  const int NP = (R + 15) & ~15;
  const uint32_t idesc_qk = umma_idesc_f16(NP, false, false);
  const uint32_t idesc_pv = umma_idesc_f16(NP, true, true);

  // ------------------------------------------------------------ producer
  if (warp == 0) {
    if (active) produce_pages<0>(p, pre, stages, full, empty, valid, flags, kTcStages, p0, p1, lane);
    return;
  }

  // ------------------------------------------------------------ converters
  if (warp <= kTcConv) {
    const int cw = warp - 1;
    TcUnits U(p, pre, p0, p1);
    bool first;
    for (int u = 0; active && U.next(first); ++u) {
      const int b = u & 1;
      bool ok = u < 2 || __all_sync(0xffffffffu, mbar_wait_bounded(&tfree[b], (uint32_t)((u >> 1) - 1) & 1u));
      uint8_t* kt = smem + L.kt + b * 32768;
      uint8_t* vt = smem + L.vt + b * 32768;
      float4* meta = reinterpret_cast<float4*>(smem + L.meta + b * 2048);
      for (int jj = 0; ok && jj < U.npg(); ++jj) {
        const int k = U.k0() + jj, s = k % kTcStages;
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[s], (uint32_t)(k / kTcStages) & 1u));
        if (!ok) break;
        const uint8_t* st4 = stages + (size_t)s * kStage4;
        const int vpage = valid[s];
        if (cw == 0 && lane == 0) vvalid[2 * b + jj] = vpage;
        if (vpage) {
          const int w = lane & 15;
#pragma unroll 4
          for (int it = 0; it < 16; ++it) {
            const int tt = 32 * cw + 2 * it + (lane >> 4);  // token of the page
            const int slot = 64 * jj + tt;                  // token of the unit
            const uint32_t kw = *reinterpret_cast<const uint32_t*>(st4 + tt * kRec4 + 4 * w);
            const uint32_t vw = *reinterpret_cast<const uint32_t*>(st4 + kPage * kRec4 + tt * kRec4 +
                                                                 16 * ((w >> 2) ^ ((tt >> 1) & 3)) + 4 * (w & 3));
            uint32_t hk[4], hv[4];
            unpack8_biased(kw, hk);
            unpack8_v(vw, hv);
            const int off = (w >> 3) * 16384 + tc_chunk(slot, w & 7);
            *reinterpret_cast<uint4*>(kt + off) = make_uint4(hk[0], hk[1], hk[2], hk[3]);
            *reinterpret_cast<uint4*>(vt + off) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
          }
          const int tt = 32 * cw + lane;
          const uint32_t* mw = reinterpret_cast<const uint32_t*>(st4 + 2 * kPage * kRec4);
          const uint32_t mk = mw[tt], mv = mw[kPage + tt];
          const float sv = h2f_lo(mv);
          meta[64 * jj + tt] = make_float4(h2f_lo(mk) * p.score_scale, h2f_hi(mk), sv, fmaf(7.5f, sv, h2f_hi(mv)));
        }
        fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
      if (!ok) {
        if (lane == 0) set_err(p.dev_err, KVQ_DEVERR_TIMEOUT);
        flags[0] = 1;
        break;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&tready[b]);
    }
    return;
  }

  // ------------------------------------------------------------ MMA warp
  if (warp == 3) {
    if (lane == 0 && active) {
      // Polls the readiness of the next QK (tiles converted, its S buffer read, Q' of a new
      // segment written) and of the oldest PV (P written, O of the previous segment read) and
      // issues whichever is ready, so neither waits behind the other.
      TcUnits Uq(p, pre, p0, p1), Up(p, pre, p0, p1);
      bool fq = false, fp = false;
      bool qmore = Uq.next(fq), pmore = Up.next(fp);
      int vq = 0, vp = 0;  // next unit to get its QK / its PV
      bool ok = true;
      uint64_t t_idle = 0;
      uint32_t idle = 0;
      while (pmore) {
        bool progressed = false;
        if (qmore) {
          const int b = vq & 1;
          if (mbar_test(&tready[b], (uint32_t)(vq >> 1) & 1u) &&
              (vq < 2 || mbar_test(&sfree[b], (uint32_t)((vq >> 1) - 1) & 1u)) &&
              (!fq || mbar_test(qready, (uint32_t)Uq.sidx & 1u))) {
            tc_fence_after();
            const uint32_t kt = smem_addr(smem + L.kt + b * 32768), qt = smem_addr(smem + L.qt);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              umma_f16(tmem + 64 * b, umma_sdesc(kt + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                       umma_sdesc(qt + (kk >> 2) * 6144 + (kk & 3) * 32, 16, 1024), idesc_qk, kk > 0);
            umma_commit(&sfull[b]);
            ++vq;
            qmore = Uq.next(fq);
            progressed = true;
          }
        }
        if (vp < vq) {
          const int b = vp & 1;
          if (mbar_test(&pready[b], (uint32_t)(vp >> 1) & 1u) &&
              (!fp || Up.sidx == 0 || mbar_test(ofree, (uint32_t)(Up.sidx - 1) & 1u))) {
            tc_fence_after();
            const uint32_t vt = smem_addr(smem + L.vt + b * 32768), pt = smem_addr(smem + L.pt + b * 16384);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              umma_f16(tmem + 128, umma_sdesc(vt + kk * 2048, 16384, 1024), umma_sdesc(pt + kk * 2048, 16384, 1024),
                       idesc_pv, (fp && kk == 0) ? 0u : 1u);
            umma_commit(&tfree[b]);
            ++vp;
            pmore = Up.next(fp);
            progressed = true;
          }
        }
        if (progressed) {  // the clock is read only every 1024 idle polls (it is slow to read)
          idle = 0;
          t_idle = 0;
        } else if ((++idle & 1023u) == 0) {
          if (t_idle == 0) {
            t_idle = globaltimer();
          } else if (globaltimer() - t_idle > kWaitLimitNs) {
            ok = false;
            break;
          }
        }
      }
      if (!ok) {
        set_err(p.dev_err, KVQ_DEVERR_TIMEOUT);
        flags[0] = 1;
      }
      umma_commit(fin);  // every MMA issued above has completed once this arrives
      if (!mbar_wait_bounded(fin, 0)) set_err(p.dev_err, KVQ_DEVERR_TIMEOUT);
    }
    __syncwarp();
    tc_fence_before();
    named_barrier(3, 32 + kTcSoft * 32);
    tc_fence_after();
    tmem_dealloc_256(tmem);
    return;
  }

  // ------------------------------------------------------------ softmax warps
  const int sw = warp - 4, q = sw & 3, rh = sw >> 2;
  const int tok = 32 * q + lane;                  // token of the unit = tensor-memory lane
  const uint32_t lane_base = (uint32_t)(32 * q) << 16;
  const int nsoft = kTcSoft * 32;
  const int tid = threadIdx.x - 4 * 32;           // 0..255
  float l[kTcHalf], ov[kTcHalf];
#pragma unroll
  for (int j = 0; j < kTcHalf; ++j) l[j] = ov[j] = 0.0f;

  // Q' tile and per-row constants of the segment of sequence bq, KV head hq
  auto load_segment = [&](int bq, int hq) {
    for (int e = tid; e < kTcMaxRows * 16; e += nsoft) {  // 16 threads per row, one 8-dim chunk each
      const int r = e >> 4, w = e & 15;
      float qv[8];
      if (r < R) {
        const float* qrow = p.q_rot + (((size_t)bq * p.S + r / G) * p.Hq + hq * G + r % G) * kD + 8 * w;
#pragma unroll
        for (int m = 0; m < 8; ++m) qv[m] = qrow[tc_dim(m) - 8 * (m >> 3)];
      } else {
#pragma unroll
        for (int m = 0; m < 8; ++m) qv[m] = 0.0f;
      }
      uint32_t hq4[4];
      float part = 0.0f, bsum = 0.0f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float hs = (i & 1) ? 0.0625f : 1.0f;  // positions 2, 3, 6, 7 meet high nibbles
        hq4[i] = pack_f16x2(qv[2 * i] * hs, qv[2 * i + 1] * hs);
        bsum += h2f_lo(hq4[i]) + h2f_hi(hq4[i]);
        part += qv[2 * i] + qv[2 * i + 1];
      }
      *reinterpret_cast<uint4*>(smem + L.qt + (w >> 3) * 6144 + tc_chunk(r, w & 7)) =
          make_uint4(hq4[0], hq4[1], hq4[2], hq4[3]);
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) {
        part += __shfl_xor_sync(0xffffffffu, part, o);
        bsum += __shfl_xor_sync(0xffffffffu, bsum, o);
      }
      if (w == 0) {
        rowc[r] = make_float4(-1024.0f * bsum, part * p.score_scale, 0.0f, -INFINITY);
        rowst[r] = -INFINITY;
      }
    }
    fence_proxy_async_shared();
  };

  TcUnits U(p, pre, p0, p1);
  bool first = false;
  bool more = active && U.next(first);
  bool err = false;
  if (more) load_segment(U.b, U.h);
  err = named_barrier_or(2, nsoft, false);
  if (more && tid == 0) mbar_arrive(qready);
  int ctxb = 0;
  bool pend = false;  // a failed wait of the previous step, reported at the next barrier
  for (int v = 0; more && !err; ++v) {
    const int b = v & 1;
    const uint32_t rb = (uint32_t)(v >> 1) & 1u;
    if (first) {
      bool bad = false;
      ctxb = eff_ctx(p, U.b, bad, 0);
    }
    bool ok = mbar_wait_bounded(&tready[b], rb) && mbar_wait_bounded(&sfull[b], rb);
    float d[kTcHalf];
    if (ok) {
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < kTcHalf / 8; ++c) {
        float t8[8];
        tmem_ld8(tmem + lane_base + 64 * b + kTcHalf * rh + 8 * c, t8);
#pragma unroll
        for (int i = 0; i < 8; ++i) d[8 * c + i] = t8[i];
      }
      tmem_wait_ld();
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&sfree[b]);

    // ---- scores of this token for rows kTcHalf * rh + j (causal limits only on a unit that
    // reaches past the context)
    const int npg = U.npg(), jj = tok >> 6;
    const bool tvalid = ok && jj < npg && vvalid[2 * b + jj] != 0;
    const int pos = (U.lp() + jj) * kPage + (tok & 63);
    const bool unit_mask = (U.lp() + npg) * kPage - 1 > ctxb;
    const float4 mt = tvalid ? reinterpret_cast<const float4*>(smem + L.meta + b * 2048)[tok]
                             : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    const bool big = mt.z >= 255.0f;
    bool need = false;
#pragma unroll
    for (int j = 0; j < kTcHalf; ++j) {
      const int r = kTcHalf * rh + j;
      float sc = -INFINITY;
      if (r < R && tvalid && (!unit_mask || pos <= ctxb + r / G)) {
        const float4 c = rowc[r];
        sc = fmaf(d[j] + c.x, mt.x, fmaf(mt.y, c.y, c.z));
        need |= sc > (big ? fminf(c.w, 0.0f) : c.w);
      }
      d[j] = sc;
    }
    if (named_barrier_or(2, nsoft, need || !ok || pend)) {
      err = named_barrier_or(2, nsoft, !ok || pend);
      if (err) break;
      // ---- rare: move the base of the rows that need it (per-row maximum over the 128 tokens)
#pragma unroll
      for (int j = 0; j < kTcHalf; ++j) {
        float mx = d[j];
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 0) rowm[sw * kTcHalf + j] = mx;
      }
      named_barrier(2, nsoft);
      bool resc = false;
      float alpha[kTcHalf];
#pragma unroll
      for (int j = 0; j < kTcHalf; ++j) {
        const int r = kTcHalf * rh + j;
        alpha[j] = 1.0f;
        if (r >= R) continue;
        float mt4 = rowm[(4 * rh) * kTcHalf + j];
        for (int qq = 1; qq < 4; ++qq) mt4 = fmaxf(mt4, rowm[(4 * rh + qq) * kTcHalf + j]);
        const float4 c = rowc[r];
        const float mold = rowst[r], muse = -c.z;
        const float mnew = fmaxf(mold, muse + mt4);
        if (mnew != mold) {
          const float mu2 = mnew == -INFINITY ? 0.0f : mnew;
          alpha[j] = fast_exp2(mold - mu2);
          d[j] += muse - mu2;
          l[j] *= alpha[j];
          ov[j] *= alpha[j];
          resc = true;
        }
      }
      // O rows of this warp's tensor-memory lanes, columns of its row half (not on a
      // segment's first unit: O starts from zero there)
      const bool any_resc = named_barrier_or(2, nsoft, resc);
      if (any_resc && !first) {
        const bool okp = mbar_wait_bounded(&tfree[b ^ 1], (uint32_t)((v - 1) >> 1) & 1u);
        if (okp) {
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < kTcHalf / 8; ++c) {
            float t8[8];
            tmem_ld8(tmem + lane_base + 128 + kTcHalf * rh + 8 * c, t8);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 8; ++i) t8[i] *= alpha[8 * c + i];
            tmem_st8(tmem + lane_base + 128 + kTcHalf * rh + 8 * c, t8);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        err = named_barrier_or(2, nsoft, !okp);
        if (err) break;
      }
      if (q == 0 && lane < kTcHalf) {  // one writer per row publishes the new base
        const int r = kTcHalf * rh + lane;
        if (r < R) {
          float mt4 = rowm[(4 * rh) * kTcHalf + lane];
          for (int qq = 1; qq < 4; ++qq) mt4 = fmaxf(mt4, rowm[(4 * rh + qq) * kTcHalf + lane]);
          const float4 c = rowc[r];
          const float mold = rowst[r];
          const float mnew = fmaxf(mold, -c.z + mt4);
          if (mnew != mold) {
            rowst[r] = mnew;
            rowc[r] = make_float4(c.x, c.y, mnew == -INFINITY ? 0.0f : -mnew, mnew == -INFINITY ? -INFINITY : 8.0f);
          }
        }
      }
      named_barrier(2, nsoft);
    }

    // ---- P and P s_V (f16, token-major) for the PV product
    uint32_t pk[kTcHalf / 2];
#pragma unroll
    for (int j = 0; j < kTcHalf; j += 2) {
      const float p0v = fast_exp2(d[j]), p1v = fast_exp2(d[j + 1]);
      l[j] += p0v;
      l[j + 1] += p1v;
      ov[j] = fmaf(p0v, mt.w, ov[j]);
      ov[j + 1] = fmaf(p1v, mt.w, ov[j + 1]);
      pk[j / 2] = pack_f16x2_sat(p0v * mt.z, p1v * mt.z);
    }
    ok = v < 2 || mbar_wait_bounded(&tfree[b], (uint32_t)((v >> 1) - 1) & 1u);
    if (ok) {
      uint8_t* pt = smem + L.pt + b * 16384;
#pragma unroll
      for (int c = 0; c < kTcHalf / 8; ++c)
        *reinterpret_cast<uint4*>(pt + tc_chunk(tok, (kTcHalf / 8) * rh + c)) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      fence_proxy_async_shared();
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&pready[b]);
    pend = !ok;

    if (U.last()) {
      // ---- segment end: token sums per row, next segment's Q', then O -> CTA partial
      const int bs = U.b, hs = U.h, seg = bs * p.Hkv + hs;
#pragma unroll
      for (int j = 0; j < kTcHalf; ++j) {
        float lt = l[j], ot = ov[j];
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
          lt += __shfl_xor_sync(0xffffffffu, lt, o);
          ot += __shfl_xor_sync(0xffffffffu, ot, o);
        }
        if (lane == 0) {
          red[(sw * kTcHalf + j) * 2] = lt;
          red[(sw * kTcHalf + j) * 2 + 1] = ot;
        }
        l[j] = ov[j] = 0.0f;
      }
      err = named_barrier_or(2, nsoft, pend);
      if (err) break;
      pend = false;
      if (q == 0 && lane < kTcHalf && kTcHalf * rh + lane < R) {
        const int r = kTcHalf * rh + lane;
        float lt = 0.0f, ot = 0.0f;
        for (int qq = 0; qq < 4; ++qq) {
          lt += red[((4 * rh + qq) * kTcHalf + lane) * 2];
          ot += red[((4 * rh + qq) * kTcHalf + lane) * 2 + 1];
        }
        float* dst = p.partials + ((size_t)(blockIdx.x + seg) * R + r) * kPartialStride;
        dst[0] = rowst[r];
        dst[1] = lt;
        ovrow[r] = ot;
      }
      named_barrier(2, nsoft);
      bool f2 = false;
      more = U.next(f2);
      if (more) load_segment(U.b, U.h);
      named_barrier(2, nsoft);
      if (more && tid == 0) mbar_arrive(qready);
      // O of the finished segment (lane = dim position, columns = rows of this half)
      ok = mbar_wait_bounded(&tfree[b], rb);
      if (ok) {
        tc_fence_after();
        float o[kTcHalf];
#pragma unroll
        for (int c = 0; c < kTcHalf / 8; ++c) {
          float t8[8];
          tmem_ld8(tmem + lane_base + 128 + kTcHalf * rh + 8 * c, t8);
#pragma unroll
          for (int i = 0; i < 8; ++i) o[8 * c + i] = t8[i];
        }
        tmem_wait_ld();
        const int m = tok, dim = tc_dim(m);
        const float us = v_unscale(dim & 3);
#pragma unroll
        for (int j = 0; j < kTcHalf; ++j) {
          const int r = kTcHalf * rh + j;
          if (r < R)
            p.partials[((size_t)(blockIdx.x + seg) * R + r) * kPartialStride + 2 + dim] = fmaf(o[j], us, ovrow[r]);
        }
      }
      tc_fence_before();
      err = named_barrier_or(2, nsoft, !ok);
      if (!err && more && tid == 0) mbar_arrive(ofree);
      first = f2;
    } else {
      more = U.next(first);
    }
  }
  if (err && tid == 0) {
    set_err(p.dev_err, KVQ_DEVERR_TIMEOUT);
    flags[0] = 1;
  }
  tc_fence_before();
  named_barrier(3, 32 + kTcSoft * 32);
}

// One block per (segment, query row): merges the segment's CTA partials and normalises.
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
  bool vattr = false;  // many-row kernel: shared-memory attribute set, occupancy cache
  bool tattr = false;  // tcgen05 many-row kernel: shared-memory attribute set
  size_t vocc_smem = 0;
  int vocc_threads = 0, vocc = 0;
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

// int4 with S x G > 8 rows: the shared-tile kernel (T = row tiles), then the same combine.
cudaError_t launch_verify(AttnParams& p, int T, long long p_max, cudaStream_t stream) {
  int dev = 0;
  cudaGetDevice(&dev);
  p.ntg = T;
  p.nkg = 1;
  p.nstages = kVStages;
  p.rows_pad = 8 * T;
  const size_t smem = VerifyLayout(p.B).total;
  const int threads = (1 + kConvWarps + T) * 32;
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
    if (!dc.vattr) {
      e = cudaFuncSetAttribute(attn_verify_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 220 * 1024);
      if (e != cudaSuccess) return e;
      dc.vattr = true;
    }
    if (dc.vocc_smem != smem || dc.vocc_threads != threads) {
      int o = 0;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, attn_verify_kernel, threads, smem);
      if (e != cudaSuccess) return e;
      dc.vocc = std::max(o, 1);
      dc.vocc_smem = smem;
      dc.vocc_threads = threads;
    }
    occ = dc.vocc;
    sm = dc.sm;
  }
  long long grid = std::min<long long>((long long)sm * occ, kMaxCtas);
  grid = std::max<long long>(1, std::min(grid, p_max));
  p.n_cta = (int)grid;
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
  e = cudaLaunchKernelEx(&cfg, attn_verify_kernel, p);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3((unsigned)(p.B * p.Hkv * p.R), 1, 1);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = (p.B + 1 + 4) * sizeof(int);
  return cudaLaunchKernelEx(&cfg, combine_kernel<0>, p);
}

// int4 with many query rows through the tcgen05 kernel, then the same combine.
cudaError_t launch_tc(AttnParams& p, long long p_max, cudaStream_t stream) {
  int dev = 0;
  cudaGetDevice(&dev);
  const size_t smem = TcLayout(p.B).total + 1024;  // + alignment of the tile atoms
  cudaError_t e = cudaSuccess;
  int sm = 1;
  {
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DevCache& dc = g_dev[(dev >= 0 && dev < 64) ? dev : 0];
    if (dc.sm == 0) {
      int n = 0;
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
      dc.sm = n > 0 ? n : 1;
    }
    if (!dc.tattr) {
      e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
      if (e != cudaSuccess) return e;
      dc.tattr = true;
    }
    sm = dc.sm;
  }
  long long grid = std::min<long long>((long long)sm, kMaxCtas);  // one CTA per SM
  grid = std::max<long long>(1, std::min(grid, p_max));
  p.n_cta = (int)grid;
  p.ntg = 1;
  p.nkg = 1;
  p.nstages = kTcStages;
  p.rows_pad = kTcMaxRows;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3((unsigned)kTcThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, attn_tc_kernel, p);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3((unsigned)(p.B * p.Hkv * p.R), 1, 1);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = (p.B + 1 + 4) * sizeof(int);
  return cudaLaunchKernelEx(&cfg, combine_kernel<0>, p);
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
  if (job.fmt == 0 && ntiles >= KVQ_VERIFY_MIN_TILES) {
    const char* sel = getenv("KVQ_MANY_ROWS_KERNEL");
    if (sel && strcmp(sel, "tcgen05") == 0) return launch_tc(p, p_max, stream);
    if (sel && strcmp(sel, "tile") == 0) return launch_verify(p, ntiles, p_max, stream);
  }
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
