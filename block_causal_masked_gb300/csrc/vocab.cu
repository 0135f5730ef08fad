// vocab.cu -- vocabulary-wide reductions of the decode step on sm_103a:
//   unmask_kernel  argmax / max-softmax-probability / LSE of every masked
//                  position's logits row, then the per-block commit rule;
//   verify_kernel  argmax (greedy or Gumbel-max) of every AR row, then the
//                  left-to-right speculative match of each sequence.
//
// Both are HBM streams: a grid of (chunk, row) CTAs streams each row once
// (bulk copies into shared memory), keeps a running (max, first argmax, Σexp)
// per thread and merges it with warp shuffles.  The chunks of one row are one
// thread-block cluster: each hands its partial to rank 0 through distributed
// shared memory, and after one cluster barrier rank 0 merges the row and
// writes its result.  The last row to finish (an acquire-release atomic
// ticket, no spinning) runs the small per-block / per-sequence decision in the
// same launch, reading one result per row.  Counters are returned to zero, so the workspace needs
// clearing only once.
#include <cuda_bf16.h>

#include <cmath>

#include "launch.h"
#include "ptx.cuh"

namespace bd {
namespace {

// Threads of a CTA: 128, or 256 where every element costs more (sampled
// scores: two logarithms per element).  Launched with blockDim.x of either;
// per-CTA arrays are sized for the larger.
constexpr int kMaxThreads = 256;
constexpr int kLightThreads = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kMaxBlock = 1024;   // positions of one block
static_assert(kMaxChunks <= 32, "one warp merges a row's chunk partials");
constexpr int kMaxVerifyL = 1024; // slots of one verified block

// Running (max, sum of exp(x - max), first index of max).
struct Acc {
  float m;
  float s;
  int idx;
};

__device__ __forceinline__ void acc_merge(Acc& a, const Acc& b) {
  if (b.m == -INFINITY) return;
  if (a.m == -INFINITY) {
    a = b;
    return;
  }
  const float M = fmaxf(a.m, b.m);
  const float s = a.s * fast_exp2((a.m - M) * kLog2e) + b.s * fast_exp2((b.m - M) * kLog2e);
  a.idx = a.m > b.m ? a.idx : (b.m > a.m ? b.idx : min(a.idx, b.idx));
  a.m = M;
  a.s = s;
}

// Folds a vector of n values starting at index i0 into the accumulator.
template <int N>
__device__ __forceinline__ void acc_vec(Acc& a, const float (&x)[N], int i0, bool need_sum) {
  float vm = x[0];
  int vi = 0;
#pragma unroll
  for (int k = 1; k < N; ++k)
    if (x[k] > vm) { vm = x[k]; vi = k; }
  if (vm > a.m) {
    if (need_sum) a.s = (a.m == -INFINITY) ? 0.f : a.s * fast_exp2((a.m - vm) * kLog2e);
    a.m = vm;
    a.idx = i0 + vi;
  }
  if (need_sum) {
#pragma unroll
    for (int k = 0; k < N; ++k) a.s += fast_exp2((x[k] - a.m) * kLog2e);
  }
}

__device__ __forceinline__ float load_one(const void* base, int dtype, long long off) {
  if (dtype == BD_BF16) {
    const unsigned short h = __ldg(reinterpret_cast<const unsigned short*>(base) + off);
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
  }
  return __ldg(static_cast<const float*>(base) + off);
}

// Gumbel-perturbed score x / T - ln(-ln u); the inner logarithm is taken with
// full precision because u close to 1 decides the largest perturbations.
__device__ __forceinline__ float gumbel_score(float x, float u, float inv_temp) {
  return fmaf(x, inv_temp, -__logf(-logf(u)));
}

// Block-wide merge of the per-thread accumulators; the result is valid in thread 0.
__device__ Acc block_reduce(Acc a, Acc* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Acc b;
    b.m = __shfl_xor_sync(0xffffffffu, a.m, o);
    b.s = __shfl_xor_sync(0xffffffffu, a.s, o);
    b.idx = __shfl_xor_sync(0xffffffffu, a.idx, o);
    acc_merge(a, b);
  }
  if (lane == 0) sh[warp] = a;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < static_cast<int>(blockDim.x) / 32; ++w) acc_merge(a, sh[w]);
  }
  return a;
}

// Pieces of a chunk are staged in shared memory by bulk copies (the copy
// engine keeps far more bytes in flight per SM than per-thread loads can), two
// pieces at a time: while one is reduced the next is landing.
constexpr int kPiece = 8192;   // elements per piece (a multiple of 8)
constexpr int kPieceStages = 2;

// Dynamic shared memory of a streaming CTA: kPieceStages pieces of logits (and
// of noise, when sampled).
__host__ __device__ constexpr int stream_smem_bytes(int elem_bytes, bool noise) {
  return kPieceStages * kPiece * (elem_bytes + (noise ? 4 : 0));
}

struct Stream {
  uint8_t* buf;     // dynamic shared memory
  uint64_t* bars;   // kPieceStages mbarriers
  int32_t* dev_status;
  uint64_t wait_ns; // limit of a wait for a piece
};

// Reduces elements [lo, hi) of one row (greedy: logits; sampled: perturbed
// scores).  Elements [lo, lo + 8 floor((hi - lo) / 8)) arrive by bulk copies
// into shared memory; a ragged tail of fewer than 8 is read directly.  Every
// copy issued has landed when this returns (the shared memory stays valid).
__device__ Acc reduce_chunk(const Stream& st, const void* logits, int dtype, long long row_off, const float* noise,
                            long long noise_off, float inv_temp, int lo, int hi, bool need_sum) {
  Acc a{-INFINITY, 0.f, 0x7fffffff};
  const int esz = dtype == BD_BF16 ? 2 : 4;
  const int stage_bytes = kPiece * (esz + (noise ? 4 : 0));
  const int vend = lo + (hi - lo) / 8 * 8;
  const int npieces = (vend - lo + kPiece - 1) / kPiece;
  int issued = 0;  // pieces issued (thread 0)
  auto issue = [&](int k) {
    ++issued;
    const int b = k % kPieceStages;
    const int e0 = lo + k * kPiece;
    const int n = min(kPiece, vend - e0);
    uint8_t* dst = st.buf + b * stage_bytes;
    mbar_arrive_expect_tx(&st.bars[b], static_cast<uint32_t>(n * (esz + (noise ? 4 : 0))));
    bulk_load(dst, static_cast<const uint8_t*>(logits) + (row_off + e0) * esz, n * esz, &st.bars[b]);
    if (noise) bulk_load(dst + kPiece * esz, noise + noise_off + e0, n * 4, &st.bars[b]);
  };
  if (threadIdx.x == 0)
    for (int k = 0; k < kPieceStages && k < npieces; ++k) issue(k);
  bool ok = true;
  for (int k = 0; k < npieces; ++k) {
    const int b = k % kPieceStages;
    const int e0 = lo + k * kPiece;
    const int nv = min(kPiece, vend - e0) / 8;
    if (ok) ok = mbar_wait_bounded(&st.bars[b], (k / kPieceStages) & 1, st.dev_status, st.wait_ns);
    if (ok) {
      const uint8_t* piece = st.buf + b * stage_bytes;
      for (int v = threadIdx.x; v < nv; v += blockDim.x) {
        float x[8];
        if (dtype == BD_BF16) {
          const uint4 w = *reinterpret_cast<const uint4*>(piece + 16 * v);
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            x[2 * q] = __uint_as_float(ws[q] << 16);
            x[2 * q + 1] = __uint_as_float(ws[q] & 0xffff0000u);
          }
        } else {
          const float4 f0 = *reinterpret_cast<const float4*>(piece + 32 * v);
          const float4 f1 = *reinterpret_cast<const float4*>(piece + 32 * v + 16);
          x[0] = f0.x; x[1] = f0.y; x[2] = f0.z; x[3] = f0.w;
          x[4] = f1.x; x[5] = f1.y; x[6] = f1.z; x[7] = f1.w;
        }
        if (noise) {
          const float4* np4 = reinterpret_cast<const float4*>(piece + kPiece * esz + 32 * v);
          const float4 n0 = np4[0], n1 = np4[1];
          const float nn[8] = {n0.x, n0.y, n0.z, n0.w, n1.x, n1.y, n1.z, n1.w};
#pragma unroll
          for (int q = 0; q < 8; ++q) x[q] = gumbel_score(x[q], nn[q], inv_temp);
        }
        acc_vec<8>(a, x, e0 + 8 * v, need_sum);
      }
    }
    __syncthreads();  // the stage is read: it may be refilled
    if (threadIdx.x == 0 && k + kPieceStages < npieces) {
      if (ok) issue(k + kPieceStages);
    }
  }
  if (threadIdx.x == 0 && !ok) {
    // a wait gave up: let the copies still in flight land before the CTA ends
    for (int k = issued > kPieceStages ? issued - kPieceStages : 0; k < issued; ++k)
      mbar_wait_bounded(&st.bars[k % kPieceStages], (k / kPieceStages) & 1, nullptr);
  }
  // ragged tail of the row (only when the row length is not a multiple of 8)
  for (int i = vend + threadIdx.x; i < hi; i += blockDim.x) {
    float x[1] = {load_one(logits, dtype, row_off + i)};
    if (noise) x[0] = gumbel_score(x[0], __ldg(noise + noise_off + i), inv_temp);
    acc_vec<1>(a, x, i, need_sum);
  }
  return a;
}

// The CTAs of one logits row are one thread-block cluster (one CTA per chunk,
// the rank = the chunk): each hands its chunk's (max, sum, first argmax) to
// rank 0 through distributed shared memory, and after one cluster barrier
// rank 0's first warp merges them, one partial per lane, into the row's result.
__device__ Acc warp_merge(const float4* parts, int chunks) {
  const int lane = threadIdx.x & 31;
  Acc a{-INFINITY, 0.f, 0x7fffffff};
  if (lane < chunks) {
    const float4 q = parts[lane];
    a = Acc{q.x, q.y, __float_as_int(q.z)};
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Acc b;
    b.m = __shfl_xor_sync(0xffffffffu, a.m, o);
    b.s = __shfl_xor_sync(0xffffffffu, a.s, o);
    b.idx = __shfl_xor_sync(0xffffffffu, a.idx, o);
    acc_merge(a, b);
  }
  return a;
}

// Hands this CTA's partial (valid in thread 0) to rank 0 of the row's cluster
// and passes the cluster barrier; in rank 0, returns the row's merged result
// (valid in thread 0).  Every thread of every CTA of the cluster calls it.
__device__ Acc cluster_row_merge(const Acc& a, float4* parts, int chunks) {
  if (threadIdx.x == 0)
    st_cluster_v4(cluster_addr(smem_addr(parts + blockIdx.x), 0), make_float4(a.m, a.s, __int_as_float(a.idx), 0.f));
  cluster_arrive();  // release: this CTA's partial is written
  cluster_wait();    // acquire: every partial of the row is in rank 0's shared memory
  Acc r{-INFINITY, 0.f, 0x7fffffff};
  if (blockIdx.x == 0 && threadIdx.x < 32) r = warp_merge(parts, chunks);
  return r;
}

constexpr int kStageRows = 2048;  // row results the deciding CTA stages in shared memory

// ======================================================================= unmask

// The commit rule, in the last CTA to finish a row: every row's result is in
// p.row_res.  `dyn` (the CTA's idle piece buffers, >= 32 KB) stages the row
// results.
__device__ void unmask_select(const UnmaskParams& p, uint8_t* dyn) {
  __shared__ uint8_t st0[kMaxPos];
  __shared__ float conf_s[kMaxPos];
  __shared__ int pred_s[kMaxPos];
  __shared__ int row_s[kMaxPos];
  __shared__ int bs_s[kMaxPos + 1];
  __shared__ int cnt[4];
  float4* res_s = reinterpret_cast<float4*>(dyn);
  const int tid = threadIdx.x;
  const int n_res = min(p.R, kStageRows);
  {
    // Every load of a thread is issued before any is used: one memory round
    // trip for the window's state, rows, partition and row results.  The
    // loops are kept rolled: this code runs once per call in one CTA, so its
    // size (instruction fetch) costs more than its instruction count.
    const int n_items = max(max(p.n_pos, p.n_blocks + 1), n_res);
#pragma unroll 1
    for (int j = tid; j < n_items; j += blockDim.x) {
      const uint8_t sv = j < p.n_pos ? p.state[j] : 0;
      const int rv = j < p.n_pos ? __ldg(p.logit_row + j) : -1;
      const int bv = j <= p.n_blocks ? __ldg(p.block_start + j) : 0;
      const float4 q = j < n_res ? __ldcg(p.row_res + j) : make_float4(0.f, 0.f, 0.f, 0.f);
      if (j < p.n_pos) {
        st0[j] = sv;
        row_s[j] = rv;
      }
      if (j <= p.n_blocks) bs_s[j] = bv;
      if (j < n_res) res_s[j] = q;
    }
  }
  __syncthreads();
  // every masked position with a logits row: prediction, confidence, LSE
#pragma unroll 1
  for (int j = tid; j < p.n_pos; j += blockDim.x) {
    const int row = row_s[j];
    int pred = -1;
    float conf = 0.f, lse = 0.f;
    if (st0[j] == BD_MASKED && row >= 0 && row < p.R) {
      const float4 q = row < kStageRows ? res_s[row] : __ldcg(p.row_res + row);
      pred = __float_as_int(q.z);
      conf = fast_rcp(q.y);
      lse = q.x + fast_log2(q.y) * kLn2;
    }
    pred_s[j] = pred;
    conf_s[j] = conf;
    if (p.pred) p.pred[j] = pred;
    if (p.conf) p.conf[j] = conf;
    if (p.lse) p.lse[j] = lse;
    p.commit[j] = 0;
  }
  int ok_local = 1;
  #pragma unroll 1
  for (int b = tid; b < p.n_blocks; b += blockDim.x) {
    const int lo = bs_s[b], hi = bs_s[b + 1];
    ok_local &= lo < hi && hi - lo <= kMaxBlock;
  }
  if (tid == 0) ok_local &= bs_s[0] == 0 && bs_s[p.n_blocks] == p.n_pos;
  if (!__syncthreads_and(ok_local)) {
    if (tid == 0 && p.dev_status) atomicOr(p.dev_status, BD_DEV_BAD_INPUT);
    return;
  }
  #pragma unroll 1
  for (int b = 0; b < p.n_blocks; ++b) {
    const int lo = bs_s[b], hi = bs_s[b + 1];
    if (tid < 4) cnt[tid] = 0;
    __syncthreads();
    int masked = 0, cand = 0, prev_done = 0;
    #pragma unroll 1
    for (int j = lo + tid; j < hi; j += blockDim.x) {
      masked += st0[j] == BD_MASKED;
      cand += pred_s[j] >= 0;
    }
    if (b > 0) {
      const int plo = bs_s[b - 1];
      #pragma unroll 1
      for (int j = plo + tid; j < lo; j += blockDim.x) prev_done += st0[j] != BD_MASKED;
    }
    // one shared-memory atomic per warp: every thread adding its own count to
    // the same word serialises them
    masked = __reduce_add_sync(0xffffffffu, masked);
    cand = __reduce_add_sync(0xffffffffu, cand);
    prev_done = __reduce_add_sync(0xffffffffu, prev_done);
    if ((tid & 31) == 0) {
      if (masked) atomicAdd(&cnt[0], masked);
      if (cand) atomicAdd(&cnt[1], cand);
      if (prev_done) atomicAdd(&cnt[2], prev_done);
    }
    __syncthreads();
    int status;
    if (cnt[0] == 0) {
      status = BD_DONE;
    } else if (b == 0) {
      status = BD_FULL;
    } else {
      const long long psize = lo - bs_s[b - 1];
      const long long done = cnt[2];
      status = done * p.act_den >= static_cast<long long>(p.act_num) * psize   ? BD_FULL
               : done * p.add_den >= static_cast<long long>(p.add_num) * psize ? BD_HALF
                                                                               : BD_INACTIVE;
    }
    const int rem = cnt[1];
    const int frac = static_cast<int>((static_cast<long long>(rem) * p.min_num + p.min_den - 1) / p.min_den);
    const int n_min = min(rem, max(p.k_fixed, frac));
    int ncom = 0;
    if (status == BD_FULL || status == BD_HALF) {
      #pragma unroll 1
      for (int j = lo + tid; j < hi; j += blockDim.x) {
        if (pred_s[j] < 0) continue;
        const float c = conf_s[j];
        bool take;
        if (status == BD_HALF) {
          take = c >= p.tau_half;
        } else {
          take = c >= p.tau_full;
          if (!take) {
            int rank = 0;
            #pragma unroll 1
            for (int k = lo; k < hi && rank < n_min; ++k)
              if (pred_s[k] >= 0 && (conf_s[k] > c || (conf_s[k] == c && k < j))) ++rank;
            take = rank < n_min;
          }
        }
        if (take) {
          p.commit[j] = 1;
          p.tokens[j] = pred_s[j];
          p.state[j] = BD_COMMITTED;
          ++ncom;
        } else if (p.write_draft) {
          p.tokens[j] = pred_s[j];
        }
      }
    } else if (p.write_draft) {
      #pragma unroll 1
      for (int j = lo + tid; j < hi; j += blockDim.x)
        if (pred_s[j] >= 0) p.tokens[j] = pred_s[j];
    }
    ncom = __reduce_add_sync(0xffffffffu, ncom);
    if ((tid & 31) == 0 && ncom) atomicAdd(&cnt[3], ncom);
    __syncthreads();
    if (tid == 0) {
      p.n_committed[b] = cnt[3];
      p.status[b] = status;
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kMaxThreads) unmask_kernel(const __grid_constant__ UnmaskParams p) {
  __shared__ Acc red[kMaxThreads / 32];
  __shared__ __align__(16) float4 parts[kMaxChunks];
  __shared__ int last;
  __shared__ __align__(8) uint64_t bars[kPieceStages];
  extern __shared__ __align__(128) uint8_t dyn[];
  if (threadIdx.x == 0) {
    for (int i = 0; i < kPieceStages; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();     // inputs may come from the previous kernel in the stream
  pdl_trigger();  // the next kernel may start its own set-up
  // one CTA per (chunk, logits row): every row is streamed, whichever position
  // it belongs to, so no lookup stands before the first load
  const int row = blockIdx.y;
  const int chunk = blockIdx.x;
  const int lo = chunk * p.chunk_elems;
  const int hi = min(p.V, lo + p.chunk_elems);
  Acc a{-INFINITY, 0.f, 0x7fffffff};
  if (lo < hi)
    a = reduce_chunk(Stream{dyn, bars, p.dev_status, p.wait_ns}, p.logits, p.dtype,
                     static_cast<long long>(row) * p.ld, nullptr, 0, 1.f, lo, hi, true);
  a = block_reduce(a, red);
  const Acc r = cluster_row_merge(a, parts, p.chunks);
  if (chunk != 0) return;
  if (threadIdx.x == 0) {
    p.row_res[row] = make_float4(r.m, r.s, __int_as_float(r.idx), 0.f);
    last = ticket_acq_rel(p.grid_ticket) == static_cast<unsigned>(p.R - 1);
  }
  __syncthreads();  // carries thread 0's acquire to the CTA
  if (!last) return;
  unmask_select(p, dyn);
  if (threadIdx.x == 0) *p.grid_ticket = 0u;
}

// ======================================================================= verify

__device__ void verify_match(const VerifyParams& p, int s) {
  __shared__ uint8_t st[kMaxVerifyL];
  __shared__ int tok[kMaxVerifyL];
  __shared__ int arg[kMaxVerifyL + 1];
  const int L = p.L;
  {
    // one memory round trip: the sequence's state, tokens and row results
    const float4* res = p.row_res + static_cast<size_t>(s) * p.n_rows;
#pragma unroll 1
    for (int j = threadIdx.x; j < max(L, p.n_rows); j += blockDim.x) {
      const uint8_t sv = j < L ? p.state[static_cast<size_t>(s) * L + j] : 0;
      const int tv = j < L ? p.tokens[static_cast<size_t>(s) * L + j] : 0;
      const float4 q = j < p.n_rows ? __ldcg(res + j) : make_float4(0.f, 0.f, 0.f, 0.f);
      if (j < L) {
        st[j] = sv;
        tok[j] = tv;
      }
      if (j < p.n_rows) arg[j] = __float_as_int(q.z) == 0x7fffffff ? -1 : __float_as_int(q.z);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int e = 0, n_acc = 0, bonus = -1, bonus_pos = -1;
    bool mismatch = false;
    #pragma unroll 1
    for (int j = 0; j < L; ++j) {
      if (st[j] == BD_SCAFFOLD) continue;
      if (st[j] == BD_MASKED) {
        if (!mismatch) {
          const int t = e < p.n_rows ? arg[e] : -1;
          if (t == tok[j]) {
            st[j] = BD_COMMITTED;
            ++n_acc;
          } else {
            tok[j] = t;
            st[j] = BD_COMMITTED;
            bonus = t;
            bonus_pos = j;
            mismatch = true;
          }
        } else {
          tok[j] = -1;
        }
      }
      ++e;
    }
    if (e + 1 != p.n_rows && p.dev_status) atomicOr(p.dev_status, BD_DEV_BAD_INPUT);
    if (!mismatch) {
      bonus = e < p.n_rows ? arg[e] : -1;
      bonus_pos = L;
    }
    p.accepted_len[s] = n_acc + 1;
    p.bonus[s] = bonus;
    p.bonus_pos[s] = bonus_pos;
  }
  __syncthreads();
  #pragma unroll 1
  for (int j = threadIdx.x; j < L; j += blockDim.x) {
    p.state[static_cast<size_t>(s) * L + j] = st[j];
    p.tokens[static_cast<size_t>(s) * L + j] = tok[j];
  }
}

__global__ void __launch_bounds__(kMaxThreads) verify_kernel(const __grid_constant__ VerifyParams p) {
  __shared__ Acc red[kMaxThreads / 32];
  __shared__ __align__(16) float4 parts[kMaxChunks];
  __shared__ int last;
  __shared__ __align__(8) uint64_t bars[kPieceStages];
  extern __shared__ __align__(128) uint8_t dyn[];
  if (threadIdx.x == 0) {
    for (int i = 0; i < kPieceStages; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.y;  // sequence * n_rows + e
  const int chunk = blockIdx.x;
  const int s = row / p.n_rows;
  const int lo = chunk * p.chunk_elems;
  const int hi = min(p.V, lo + p.chunk_elems);
  Acc a{-INFINITY, 0.f, 0x7fffffff};
  if (lo < hi)
    a = reduce_chunk(Stream{dyn, bars, p.dev_status, p.wait_ns}, p.logits, p.dtype, static_cast<long long>(row) * p.ld,
                     p.noise, static_cast<long long>(row) * p.ld, p.inv_temp, lo, hi, false);
  a = block_reduce(a, red);
  const Acc r = cluster_row_merge(a, parts, p.chunks);
  if (chunk != 0) return;
  if (threadIdx.x == 0) {
    p.row_res[row] = make_float4(r.m, 0.f, __int_as_float(r.idx), 0.f);
    last = ticket_acq_rel(p.seq_ticket + s) == static_cast<unsigned>(p.n_rows - 1);
  }
  __syncthreads();  // carries thread 0's acquire to the CTA
  if (!last) return;
  verify_match(p, s);
  if (threadIdx.x == 0) p.seq_ticket[s] = 0u;
}

}  // namespace

void vocab_split(int rows, int V, int num_sms, int* chunks, int* chunk_elems, int max_chunks) {
  // about two CTAs per SM over the whole grid, chunks of at least 2048
  // elements, at most one cluster's worth per row
  const int target = 2 * num_sms;
  int c = (target + rows - 1) / rows;
  const int max_c = (V + 2047) / 2048;
  if (c > max_c) c = max_c;
  if (c > max_chunks) c = max_chunks;
  if (c < 1) c = 1;
  int e = (V + c - 1) / c;
  e = (e + 7) / 8 * 8;
  c = (V + e - 1) / e;
  *chunks = c;
  *chunk_elems = e;
}

static size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Counter words sit in a fixed-size region at the start of the workspace, so a
// buffer reused for calls of other shapes finds them where the previous call
// left them: at zero.
size_t unmask_counter_bytes() { return 256; }
size_t verify_counter_bytes() { return align256(sizeof(unsigned) * kMaxVerifySeqs); }

size_t unmask_workspace_bytes(int R) { return unmask_counter_bytes() + align256(sizeof(float4) * static_cast<size_t>(R)); }

size_t verify_workspace_bytes(int n_seq, int n_rows) {
  return verify_counter_bytes() + align256(sizeof(float4) * static_cast<size_t>(n_seq) * n_rows);
}

// Launch with programmatic stream serialisation, so that the kernel's set-up can
// overlap the tail of the previous kernel (each kernel waits for it with
// griddepcontrol.wait before touching global memory), as clusters of the
// `chunks` CTAs of one logits row.  A cluster wider than the portable 8 needs
// that many CTAs' room in one GPC; if the device has none, the rows are cut
// into 8 chunks instead.
template <typename P>
static cudaError_t launch_rows(void (*kernel)(P), int rows, P p, int V, int smem, int threads, cudaStream_t stream) {
  static PerDeviceOnce configured;  // one instantiation per kernel
  const cudaError_t ce = configured.run([&] {
    cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, stream_smem_bytes(4, true));
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
  });
  if (ce != cudaSuccess) return ce;
  cudaLaunchConfig_t cfg = {};
  cfg.dynamicSmemBytes = smem;
  cfg.blockDim = dim3(threads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  for (;;) {
    cfg.gridDim = dim3(p.chunks, rows);
    attr[1].val.clusterDim.x = p.chunks;
    if (p.chunks <= 8) break;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) == cudaSuccess && n > 0) break;
    (void)cudaGetLastError();
    int sms = 152;
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) (void)cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    vocab_split(rows, V, sms, &p.chunks, &p.chunk_elems, 8);
  }
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, p);
  return e == cudaSuccess ? cudaGetLastError() : e;
}

cudaError_t launch_unmask(const UnmaskParams& p, cudaStream_t stream) {
  return launch_rows(unmask_kernel, p.R, p, p.V, stream_smem_bytes(p.dtype == BD_BF16 ? 2 : 4, false), kLightThreads,
                     stream);
}

cudaError_t launch_verify(const VerifyParams& p, cudaStream_t stream) {
  return launch_rows(verify_kernel, p.n_seq * p.n_rows, p, p.V,
                     stream_smem_bytes(p.dtype == BD_BF16 ? 2 : 4, p.noise != nullptr),
                     p.noise != nullptr ? kMaxThreads : kLightThreads, stream);
}

}  // namespace bd
