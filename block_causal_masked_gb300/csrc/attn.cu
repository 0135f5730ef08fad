// attn.cu -- block-causal attention and the shared-prefix fork on sm_103a.
//
// What is computed (Fast-dVLA paper notes, "关键设计 1. 分块因果注意力";
// Fast-dDrive method summary §3.1; WAM-Diff2 write-up §2.1): a query of block b
// sees every cached prefix key, every key of an earlier block and every key of
// its own block.  Because blocks are contiguous, that is "key index < a per-row
// limit": lim(i) = C + end of i's block.  The fork (Fast-dDrive method summary
// §3.3) adds N rollouts that each own private rows after one shared prefix.
//
// How (one CTA per (KV split, 128 packed query rows, KV head)):
//   * GQA rows of one KV head are packed: row = (rollout * n_q + i) * G + g, so
//     one tcgen05.mma with M = 128 serves G query heads of up to 128/G positions;
//   * warp 0 streams 128-key K and V tiles with TMA (128-byte swizzle) into a
//     two-stage ring; the prefix tiles come from one shared tensor map and are
//     reused by every packed row, private tiles from a per-rollout map;
//   * warp 1 allocates TMEM and issues S = Q·Kᵀ (into one of two TMEM S buffers)
//     and O += P·V (O stays in TMEM for the whole KV range), one thread;
//   * warps 2-5 own one TMEM lane (= one packed row) each thread: masked online
//     softmax in fp32 from TMEM, P rounded to bf16 into a swizzled smem tile;
//     the running max is only moved (and O rescaled in TMEM) when it grows by
//     more than 2^8, so most tiles need no O round trip;
//   * with RoPE, warps 6-9 rotate each staged prefix K tile in shared memory at
//     k_pos - delta before the MMA warp may read it (FlashDrive tutorial,
//     "流式推理"); the angle is reduced exactly in 0.64 fixed-point turns;
//   * KV splits write normalised fp32 partials and an LSE per row; a second
//     kernel merges them with LSE weights.
// Every wait is bounded (ptx.cuh); there is no wait on another CTA.
#include <cuda_bf16.h>

#include <cmath>

#include "launch.h"
#include "ptx.cuh"

namespace bd {
namespace {

constexpr int BM = kAttnBM;
constexpr int BN = kAttnBN;
constexpr int kStages = 2;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;  // keep a stale running max while the tile max is within 2^8

struct TileEntry {
  int32_t rollout;  // -1: shared prefix tile
  int32_t key0;     // first key of the tile within its segment
};

enum Bar : int {
  KFULL = 0, VFULL = 2, KVEMPTY = 4, SFULL = 6, SFREE = 8, PFULL = 10, ODONE = 11, QFULL = 12,
  KREADY = 13, DRAIN = 15, NUM_BARS = 16
};

template <int D>
struct Layout {
  static constexpr int kQBytes = BM * D * 2;
  static constexpr int kKVBytes = BN * D * 2;  // one K or one V tile
  static constexpr int kPBytes = BM * BN * 2;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kQBytes;
  static constexpr int kV = kK + kStages * kKVBytes;
  static constexpr int kP = kV + kStages * kKVBytes;
  static constexpr int kBar = kP + kPBytes;
  static constexpr int kTiles = kBar + NUM_BARS * 8;
  static constexpr int kMisc = kTiles + kAttnMaxTiles * 8;
  static constexpr int kEnd = kMisc + 64;
  static constexpr int kAlloc = kEnd + 1024;  // slack to align the base to 1024 B
  // TMEM columns: S buffers [0, 2*BN), O [2*BN, 2*BN + D)
  static constexpr uint32_t kTmemCols = 512;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t a = smem_addr(p);
  return p + (((a + 1023u) & ~1023u) - a);
}

__device__ __forceinline__ bool all_lanes(bool v) { return __all_sync(0xffffffffu, v); }

// Same as mbar_wait but ignores the abort flag: used to let copies and MMAs in
// flight finish before the CTA releases its shared memory and TMEM.
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity, int32_t* dev_status) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > kWaitLimitNs) {
      if (dev_status) atomicOr(dev_status, BD_DEV_TIMEOUT);
      return;
    }
  }
}

// End (exclusive) of the block that holds active position i, clamped to [1, n_q].
__device__ __forceinline__ int block_end_of(const AttnParams& p, int i) {
  int e;
  if (p.block_start == nullptr) {
    e = (i / p.block_size + 1) * p.block_size;
  } else {
    int lo = 0, hi = p.n_blocks - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(p.block_start + mid) <= i) lo = mid; else hi = mid - 1;
    }
    e = __ldg(p.block_start + lo + 1);
  }
  return max(1, min(p.n_q, e));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ void bf16x2_unpack(uint32_t w, float& lo, float& hi) {
  lo = __uint_as_float(w << 16);
  hi = __uint_as_float(w & 0xffff0000u);
}

// cos/sin of pos * freq_d with freq_d / (2 pi) given as a 0.64 fixed-point
// fraction: the product modulo 2^64 is the fractional turn, so the reduction
// to [-pi, pi) is exact up to the 2^-32 truncation of its top word.
__device__ __forceinline__ void rope_cos_sin(int pos, unsigned long long turns, float& c, float& s) {
  const unsigned long long prod = static_cast<unsigned long long>(static_cast<long long>(pos)) * turns;
  const int top = static_cast<int>(prod >> 32);
  const float ang = static_cast<float>(top) * (6.283185307179586f / 4294967296.0f);
  __sincosf(ang, &s, &c);
}

// Builds this CTA's list of K/V tiles (prefix tiles, then the private tiles of
// every rollout its rows belong to, up to the furthest key any of them sees)
// and keeps the contiguous share of split `split`.  Returns the count.
__device__ int build_tiles(const AttnParams& p, int m0, int split, TileEntry* tiles) {
  if (p.block_start != nullptr) {
    bool ok = __ldg(p.block_start) == 0 && __ldg(p.block_start + p.n_blocks) == p.n_q;
    for (int b = 0; ok && b < p.n_blocks; ++b) ok = __ldg(p.block_start + b) < __ldg(p.block_start + b + 1);
    if (!ok) {
      if (p.dev_status) atomicOr(p.dev_status, BD_DEV_BAD_INPUT);
      return 0;
    }
  }
  const int per_roll = p.n_q * p.G;
  const int row_end = min(m0 + BM, p.rows_per_head);
  const int r_first = m0 / per_roll;
  const int r_last = (row_end - 1) / per_roll;
  int total = 0;
  for (int j = 0; j < p.n_prefix_tiles && total < kAttnMaxTiles; ++j) tiles[total++] = {-1, j * BN};
  for (int r = r_first; r <= r_last; ++r) {
    const int row_hi = min(row_end, (r + 1) * per_roll) - 1;
    const int i_hi = (row_hi - r * per_roll) / p.G;
    const int lim = p.priv_len + block_end_of(p, i_hi);
    for (int k0 = 0; k0 < lim && total < kAttnMaxTiles; k0 += BN) tiles[total++] = {r, k0};
  }
  const int lo = static_cast<int>(static_cast<long long>(split) * total / p.num_splits);
  const int hi = static_cast<int>(static_cast<long long>(split + 1) * total / p.num_splits);
  for (int t = lo; t < hi; ++t) tiles[t - lo] = tiles[t];
  return hi - lo;
}

template <int D, bool ROPE>
__global__ void __launch_bounds__(ROPE ? 320 : 192, 1)
    attn_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ AttnMaps maps) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  TileEntry* tiles = reinterpret_cast<TileEntry*>(smem + L::kTiles);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::kMisc);  // [0] tmem base, [1] abort, [2] tiles
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int split = blockIdx.x;
  const int m0 = blockIdx.y * BM;
  const int kvh = blockIdx.z;
  int32_t* ds = p.dev_status;

  if (threadIdx.x == 0) {
    mbar_init(&bars[KFULL + 0], 1);
    mbar_init(&bars[KFULL + 1], 1);
    mbar_init(&bars[VFULL + 0], 1);
    mbar_init(&bars[VFULL + 1], 1);
    mbar_init(&bars[KVEMPTY + 0], 1);
    mbar_init(&bars[KVEMPTY + 1], 1);
    mbar_init(&bars[SFULL + 0], 1);
    mbar_init(&bars[SFULL + 1], 1);
    mbar_init(&bars[SFREE + 0], 128);
    mbar_init(&bars[SFREE + 1], 128);
    mbar_init(&bars[PFULL], 128);
    mbar_init(&bars[ODONE], 1);
    mbar_init(&bars[QFULL], 128);
    mbar_init(&bars[KREADY + 0], 128);
    mbar_init(&bars[KREADY + 1], 128);
    mbar_init(&bars[DRAIN], 1);
    misc[1] = 0;
    misc[2] = static_cast<uint32_t>(build_tiles(p, m0, split, tiles));
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&misc[0], L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  const int nt = static_cast<int>(misc[2]);

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0 && nt > 0) {
      if (p.n_prefix_tiles > 0) { tma_prefetch_desc(&maps.pk); tma_prefetch_desc(&maps.pv); }
      tma_prefetch_desc(&maps.rk);
      tma_prefetch_desc(&maps.rv);
      int last[2] = {-1, -1};
      for (int t = 0; t < nt; ++t) {
        const int s = t & 1;
        if (t >= 2 && !mbar_wait(&bars[KVEMPTY + s], ((t >> 1) - 1) & 1, abort_flag, ds)) break;
        const TileEntry te = tiles[t];
        uint8_t* kdst = smem + L::kK + s * L::kKVBytes;
        uint8_t* vdst = smem + L::kV + s * L::kKVBytes;
        mbar_arrive_expect_tx(&bars[KFULL + s], L::kKVBytes);
#pragma unroll
        for (int hh = 0; hh < D / 64; ++hh) {
          if (te.rollout < 0)
            tma_load_3d(kdst + hh * BN * 128, &maps.pk, hh * 64, te.key0, kvh, &bars[KFULL + s]);
          else
            tma_load_4d(kdst + hh * BN * 128, &maps.rk, hh * 64, te.key0, kvh, te.rollout, &bars[KFULL + s]);
        }
        mbar_arrive_expect_tx(&bars[VFULL + s], L::kKVBytes);
#pragma unroll
        for (int hh = 0; hh < D / 64; ++hh) {
          if (te.rollout < 0)
            tma_load_3d(vdst + hh * BN * 128, &maps.pv, hh * 64, te.key0, kvh, &bars[VFULL + s]);
          else
            tma_load_4d(vdst + hh * BN * 128, &maps.rv, hh * 64, te.key0, kvh, te.rollout, &bars[VFULL + s]);
        }
        last[s] = t;
      }
      for (int s = 0; s < 2; ++s) {
        if (last[s] < 0) continue;
        mbar_drain(&bars[KFULL + s], (last[s] >> 1) & 1, ds);
        mbar_drain(&bars[VFULL + s], (last[s] >> 1) & 1, ds);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0 && nt > 0) {
      constexpr uint32_t kIdS = mma_idesc_bf16(BM, BN, false);
      constexpr uint32_t kIdPV = mma_idesc_bf16(BM, D, true);
      const uint32_t qa = smem_addr(smem + L::kQ);
      const uint32_t pa = smem_addr(smem + L::kP);
      auto issue_s = [&](int u) -> bool {
        const int s = u & 1;
        uint64_t* kb = ROPE ? &bars[KREADY + s] : &bars[KFULL + s];
        if (!mbar_wait(kb, (u >> 1) & 1, abort_flag, ds)) return false;
        if (u >= 2 && !mbar_wait(&bars[SFREE + s], ((u >> 1) - 1) & 1, abort_flag, ds)) return false;
        tc_fence_after();
        const uint32_t ka = smem_addr(smem + L::kK + s * L::kKVBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t qoff = (kk >> 2) * (BM * 128) + (kk & 3) * 32;
          const uint32_t koff = (kk >> 2) * (BN * 128) + (kk & 3) * 32;
          mma_bf16(tmem + s * BN, sw128_desc(qa + qoff, 16, 1024), sw128_desc(ka + koff, 16, 1024), kIdS,
                   kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars[SFULL + s]);
        return true;
      };
      bool ok = mbar_wait(&bars[QFULL], 0, abort_flag, ds);
      if (ok) {
        tc_fence_after();
        ok = issue_s(0);
      }
      for (int t = 0; ok && t < nt; ++t) {
        if (t + 1 < nt && !issue_s(t + 1)) break;
        if (!mbar_wait(&bars[PFULL], t & 1, abort_flag, ds)) break;
        if (!mbar_wait(&bars[VFULL + (t & 1)], (t >> 1) & 1, abort_flag, ds)) break;
        tc_fence_after();
        const uint32_t va = smem_addr(smem + L::kV + (t & 1) * L::kKVBytes);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          const uint32_t poff = (kk >> 2) * (BM * 128) + (kk & 3) * 32;
          const uint32_t voff = kk * 16 * 128;
          mma_bf16(tmem + 2 * BN, sw128_desc(pa + poff, 16, 1024), sw128_desc(va + voff, BN * 128, 1024),
                   kIdPV, (t > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&bars[ODONE]);
        mma_commit(&bars[KVEMPTY + (t & 1)]);
      }
      mma_commit(&bars[DRAIN]);
      mbar_drain(&bars[DRAIN], 0, ds);
    }
  } else if (warp < 6) {
    // ---------------------------------------------------------------- softmax rows
    const int quad = warp & 3;
    const int rl = quad * 32 + lane;  // TMEM lane = packed row within the tile
    const int row = m0 + rl;
    const int per_roll = p.n_q * p.G;
    const bool valid = row < p.rows_per_head;
    int r_row = 0, i_row = 0, g = 0;
    if (valid) {
      r_row = row / per_roll;
      const int rem = row - r_row * per_roll;
      i_row = rem / p.G;
      g = rem - i_row * p.G;
    }
    const int qhead = kvh * p.G + g;
    const size_t orow = (static_cast<size_t>(r_row) * p.n_q + i_row) * p.Hq + qhead;
    {
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.q) + orow * D);
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const uint4 val = valid ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(smem + L::kQ + sw128_offset(rl, c * 8, BM)) = val;
      }
    }
    fence_proxy_async_smem();
    mbar_arrive(&bars[QFULL]);

    const int lim_priv = valid ? p.priv_len + block_end_of(p, i_row) : 0;
    const bool warp_active = __any_sync(0xffffffffu, valid);
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    float m_run = -INFINITY;  // running max, log2-scaled
    float l_run = 0.f;
    bool ok = true;
    float v[32];
    for (int t = 0; t < nt; ++t) {
      const int s = t & 1;
      ok = all_lanes(mbar_wait(&bars[SFULL + s], (t >> 1) & 1, abort_flag, ds));
      if (!ok) break;
      tc_fence_after();
      const TileEntry te = tiles[t];
      int lim = te.rollout < 0 ? p.C : (te.rollout == r_row ? lim_priv : 0);
      if (!valid) lim = 0;
      const int nv = max(0, min(BN, lim - te.key0));
      float mx = -INFINITY;
      if (warp_active) {
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) {
          tmem_ld32(lane_base + s * BN + c * 32, v);
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (c * 32 + j < nv) mx = fmaxf(mx, v[j]);
        }
      }
      const float m_tile = nv > 0 ? mx * p.scale_log2 : -INFINITY;
      if (t > 0) {
        ok = all_lanes(mbar_wait(&bars[ODONE], (t - 1) & 1, abort_flag, ds));
        if (!ok) break;
        tc_fence_after();
      }
      const bool grow = m_tile > -INFINITY && (m_run == -INFINITY || m_tile > m_run + kRescaleLog2);
      float alpha = 1.f;
      if (grow) {
        alpha = (m_run == -INFINITY) ? 0.f : exp2f(m_run - m_tile);
        m_run = m_tile;
        l_run *= alpha;
      }
      if (warp_active && t > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          tmem_ld32(lane_base + 2 * BN + c * 32, v);
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] *= alpha;
          tmem_st32(lane_base + 2 * BN + c * 32, v);
        }
      }
      if (warp_active) {
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) {
          tmem_ld32(lane_base + s * BN + c * 32, v);
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int k = c * 32 + 2 * j;
            const float a = k < nv ? exp2f(fmaf(v[2 * j], p.scale_log2, -m_run)) : 0.f;
            const float b = k + 1 < nv ? exp2f(fmaf(v[2 * j + 1], p.scale_log2, -m_run)) : 0.f;
            l_run += a + b;
            pk[j] = pack_bf16x2(a, b);
          }
#pragma unroll
          for (int qq = 0; qq < 4; ++qq)
            *reinterpret_cast<uint4*>(smem + L::kP + sw128_offset(rl, c * 32 + qq * 8, BM)) =
                make_uint4(pk[4 * qq], pk[4 * qq + 1], pk[4 * qq + 2], pk[4 * qq + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(&bars[SFREE + s]);
      fence_proxy_async_smem();
      mbar_arrive(&bars[PFULL]);
    }
    if (ok && nt > 0) {
      ok = all_lanes(mbar_wait(&bars[ODONE], (nt - 1) & 1, abort_flag, ds));
      tc_fence_after();
    }
    const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
    const float lse_v = l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
    const size_t total_rows = static_cast<size_t>(p.N) * p.n_q * p.Hq;
    if (warp_active) {
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        if (ok && nt > 0) {
          tmem_ld32(lane_base + 2 * BN + c * 32, v);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = 0.f;
        }
        if (!valid) continue;
        if (p.num_splits == 1) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + orow * D + c * 32);
#pragma unroll
          for (int qq = 0; qq < 4; ++qq)
            dst[qq] = make_uint4(pack_bf16x2(v[8 * qq + 0] * inv_l, v[8 * qq + 1] * inv_l),
                                 pack_bf16x2(v[8 * qq + 2] * inv_l, v[8 * qq + 3] * inv_l),
                                 pack_bf16x2(v[8 * qq + 4] * inv_l, v[8 * qq + 5] * inv_l),
                                 pack_bf16x2(v[8 * qq + 6] * inv_l, v[8 * qq + 7] * inv_l));
        } else {
          float4* dst = reinterpret_cast<float4*>(p.part_o + (split * total_rows + orow) * D + c * 32);
#pragma unroll
          for (int qq = 0; qq < 8; ++qq)
            dst[qq] = make_float4(v[4 * qq] * inv_l, v[4 * qq + 1] * inv_l, v[4 * qq + 2] * inv_l,
                                  v[4 * qq + 3] * inv_l);
        }
      }
    }
    if (valid) {
      if (p.num_splits == 1) {
        if (p.lse) p.lse[(static_cast<size_t>(r_row) * p.Hq + qhead) * p.n_q + i_row] = lse_v;
      } else {
        p.part_lse[split * total_rows + orow] = lse_v;
      }
    }
  } else if (ROPE) {
    // ---------------------------------------------------------------- RoPE on staged prefix keys
    const int kr = threadIdx.x - 192;  // key row of the tile
    for (int t = 0; t < nt; ++t) {
      const int s = t & 1;
      if (!mbar_wait(&bars[KFULL + s], (t >> 1) & 1, abort_flag, ds)) break;
      const TileEntry te = tiles[t];
      const int key = te.key0 + kr;
      if (te.rollout < 0 && key < p.C) {
        const int pos = (p.k_pos ? __ldg(p.k_pos + key) : key) - p.delta;
        uint8_t* kt = smem + L::kK + s * L::kKVBytes;
#pragma unroll 1
        for (int c = 0; c < D / 16; ++c) {
          uint4* a4 = reinterpret_cast<uint4*>(kt + sw128_offset(kr, c * 8, BN));
          uint4* b4 = reinterpret_cast<uint4*>(kt + sw128_offset(kr, c * 8 + D / 2, BN));
          uint4 xa = *a4, xb = *b4;
          uint32_t* wa = reinterpret_cast<uint32_t*>(&xa);
          uint32_t* wb = reinterpret_cast<uint32_t*>(&xb);
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            float a0, a1, b0, b1, c0, s0, c1, s1;
            bf16x2_unpack(wa[w], a0, a1);
            bf16x2_unpack(wb[w], b0, b1);
            rope_cos_sin(pos, p.rope_turns[c * 8 + 2 * w], c0, s0);
            rope_cos_sin(pos, p.rope_turns[c * 8 + 2 * w + 1], c1, s1);
            wa[w] = pack_bf16x2(a0 * c0 - b0 * s0, a1 * c1 - b1 * s1);
            wb[w] = pack_bf16x2(b0 * c0 + a0 * s0, b1 * c1 + a1 * s1);
          }
          *a4 = xa;
          *b4 = xb;
        }
        fence_proxy_async_smem();
      }
      mbar_arrive(&bars[KREADY + s]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

// Merges the KV splits of every output row: LSE = ln Σ_s exp(lse_s),
// O = Σ_s exp(lse_s - LSE) O_s.  One warp per (rollout, position, query head).
template <int D>
__global__ void __launch_bounds__(256) attn_combine_kernel(const __grid_constant__ AttnParams p) {
  const int total = p.N * p.n_q * p.Hq;
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= total) return;
  const int S = p.num_splits;
  float mx = -INFINITY;
  for (int s = lane; s < S; s += 32) mx = fmaxf(mx, p.part_lse[static_cast<size_t>(s) * total + row]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float sum = 0.f;
  for (int s = lane; s < S; s += 32) {
    const float l = p.part_lse[static_cast<size_t>(s) * total + row];
    if (l > -INFINITY) sum += exp2f((l - mx) * kLog2e);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const float LSE = mx + logf(sum);
  constexpr int E = D / 32;  // elements per lane
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  for (int s = 0; s < S; ++s) {
    const float l = p.part_lse[static_cast<size_t>(s) * total + row];
    if (!(l > -INFINITY)) continue;
    const float w = exp2f((l - LSE) * kLog2e);
    const float* src = p.part_o + (static_cast<size_t>(s) * total + row) * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      const float2 x = *reinterpret_cast<const float2*>(src + e);
      acc[e] = fmaf(w, x.x, acc[e]);
      acc[e + 1] = fmaf(w, x.y, acc[e + 1]);
    }
  }
  uint32_t* dst = reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(p.o) + static_cast<size_t>(row) * D +
                                              lane * E);
#pragma unroll
  for (int e = 0; e < E; e += 2) dst[e / 2] = pack_bf16x2(acc[e], acc[e + 1]);
  if (lane == 0 && p.lse) {
    const int ri = row / p.Hq, qhead = row - ri * p.Hq;
    const int r = ri / p.n_q, i = ri - r * p.n_q;
    p.lse[(static_cast<size_t>(r) * p.Hq + qhead) * p.n_q + i] = LSE;
  }
}

template <int D, bool ROPE>
cudaError_t launch_attn_t(const AttnParams& p, const AttnMaps& maps, int m_tiles, cudaStream_t stream) {
  static bool configured = false;
  const int smem = attn_smem_bytes(D);
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attn_kernel<D, ROPE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const dim3 grid(p.num_splits, m_tiles, p.Hkv);
  attn_kernel<D, ROPE><<<grid, ROPE ? 320 : 192, smem, stream>>>(p, maps);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.num_splits == 1) return e;
  const int total = p.N * p.n_q * p.Hq;
  attn_combine_kernel<D><<<(total + 7) / 8, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

int attn_smem_bytes(int D) {
  // D = 64 is padded so that one CTA (and its 512 TMEM columns) fills an SM.
  return D == 128 ? Layout<128>::kAlloc : (Layout<64>::kAlloc > 120 * 1024 ? Layout<64>::kAlloc : 120 * 1024);
}

cudaError_t launch_attention(const AttnParams& p, const AttnMaps& maps, int m_tiles, cudaStream_t stream) {
  if (p.D == 128) return p.rope ? launch_attn_t<128, true>(p, maps, m_tiles, stream)
                                : launch_attn_t<128, false>(p, maps, m_tiles, stream);
  return p.rope ? launch_attn_t<64, true>(p, maps, m_tiles, stream)
                : launch_attn_t<64, false>(p, maps, m_tiles, stream);
}

}  // namespace bd
