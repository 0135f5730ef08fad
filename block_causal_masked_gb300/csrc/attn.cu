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
//     three-stage K ring (a stage is refilled as soon as S of its tile is done)
//     and a two-stage V ring; the prefix tiles come from one shared tensor map
//     and are reused by every packed row, private tiles from a per-rollout map;
//   * warp 1 allocates TMEM and issues S = Q·Kᵀ (into one of two TMEM S buffers)
//     and O += P·V (P read from TMEM, O resident in TMEM for the whole KV
//     range), one thread;
//   * warps 2-9, two per TMEM lane quadrant, each hold half of the key columns
//     of their 32 packed rows: masked online softmax in fp32 from TMEM, P
//     rounded to bf16 and written back into its own S buffer; the running max
//     is only moved (and O rescaled in TMEM) when it grows by more than 2^8;
//   * the KV splits of one (row tile, KV head) form a thread-block cluster; at
//     the end every softmax thread writes its row's normalised O and (max,
//     sum) for the CTA that owns the row, one cluster barrier makes them
//     visible, and each CTA merges 1/S of the rows from all splits and stores
//     them -- one kernel, no second launch.
// With RoPE (FlashDrive tutorial, "流式推理"), the cached prefix keys stay
// pre-RoPE in memory and a small kernel of the same call rotates them at
// k_pos - delta into a bf16 copy that every row tile then reads -- once per
// call instead of once per row tile; each rotated element is the bf16 rounding
// of the rotation formed in float64 (an fp32 rotation with an error bound,
// recomputed in float64 where that bound leaves the rounding open).
// Every mbarrier wait is bounded (ptx.cuh); the only cross-CTA waits are the
// hardware cluster barriers, which every CTA of the cluster reaches on every
// path.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <climits>
#include <cmath>
#include <mutex>
#include <type_traits>

#include "launch.h"
#include "ptx.cuh"
#include "rope_table.h"

namespace bd {
namespace {

constexpr int BM = kAttnBM;
constexpr int BN = kAttnBN;
constexpr int kKStages = 3;  // K ring: a stage is free once S = Q.K^T of its tile is done (2 with FP8 K/V)
constexpr int kVStages = 2;  // V ring: a stage is free once P.V of its tile is done
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;  // keep a stale running max while the tile max is within 2^8
// warps: 0 TMA producer, 1 MMA issuer, 2..2+kSmWarps softmax
constexpr int kSmWarps = 8;
// FP8 (E4M3) K/V: two more warps dequantise the tiles, staged by TMA in a ring
// of kStgStages byte tiles, into the fp16 K / V rings
constexpr int kConvWarps = 2;
constexpr int kConvThreads = 32 * kConvWarps;
constexpr int kStgStages = 3;
template <bool KV8>
constexpr int threads_of() { return 32 * (2 + kSmWarps + (KV8 ? kConvWarps : 0)); }

struct TileEntry {
  int rollout;  // -1: shared prefix tile
  int key0;     // first key of the tile within its segment
};


enum Bar : int {
  // PFULL / ODONE: two each, by tile parity (tile t uses PFULL + t % 2 and
  // ODONE + t % 2), so that the softmax may run one tile ahead of P.V
  KFULL = 0, VFULL = 3, KEMPTY = 5, VEMPTY = 8, SFULL = 10, PFULL = 12, ODONE = 14, QFULL = 16,
  DRAIN = 17, MERGE_O = 18,
  // FP8 K/V: queries converted to fp16; staging ring of E4M3 tiles
  QCONV = 19, STG_FULL = 20, STG_EMPTY = 23, NUM_BARS = 26
};

template <int D, bool KV8 = false>
struct Layout {
  static constexpr int kKSt = KV8 ? 2 : kKStages;  // K ring stages
  static constexpr int kQBytes = BM * D * 2;
  static constexpr int kKVBytes = BN * D * 2;  // one K or one V tile (16-bit elements)
  static constexpr int kStgBytes = BN * D;     // one E4M3 tile
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kQBytes;
  static constexpr int kV = kK + kKSt * kKVBytes;
  static constexpr int kRingEnd = kV + kVStages * kKVBytes;
  static constexpr int kStg = kRingEnd;
  static constexpr int kBar = kStg + (KV8 ? kStgStages * kStgBytes : 0);
  static constexpr int kMisc = kBar + NUM_BARS * 8;
  // the two halves of a row trade tile maxima ([2 parities][2 halves][BM])
  // and final sums ([2 halves][BM])
  static constexpr int kXch = kMisc + 64;
  // (max, sum) of this CTA's rows from every split of the cluster, written by
  // the other CTAs through distributed shared memory: [S][r] float2
  static constexpr int kMLRecv = kXch + 6 * BM * 4;
  static constexpr int kEnd = kMLRecv + (BM + 2 * kAttnMaxSplits) * 8;
  // split-KV merge, over the K / V rings (idle by then): the S bf16 O
  // slices of this CTA's rows (S * r <= BM + 2 * S rows)
  static constexpr int kRecv = kK;
  static_assert(kRecv + (BM + 2 * kAttnMaxSplits) * D * 2 <= kRingEnd, "merge slices must fit");
  static constexpr int kAlloc = kEnd + 1024;  // slack to align the base to 1024 B
  static_assert(kAlloc <= 227 * 1024, "shared memory of one CTA");
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
  (void)mbar_wait_bounded(bar, parity, dev_status);
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

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ void bf16x2_unpack(uint32_t w, float& lo, float& hi) {
  lo = __uint_as_float(w << 16);
  hi = __uint_as_float(w & 0xffff0000u);
}

// ------------------------------------------------------------------ RoPE rounding
//
// The rotated key is an operand of the bf16 Q.K^T product, so it is rounded to
// bf16 -- and it must be the rounding of the rotation the definition gives:
// y = a cos(phi) - b sin(phi) (and b cos(phi) + a sin(phi)) at phi = pos * f_d,
// f_d = theta^(-2d/D), formed in float64 like the definition's arithmetic.  The
// fast path rotates in fp32 with an error bound E on |y_fp32 - y|; when the
// interval [y_fp32 - E, y_fp32 + E] holds no bf16 rounding midpoint, every
// value in it -- y included -- rounds to the same bf16, which is taken.  The
// few pairs whose interval straddles a midpoint (about 1.6e-3 of them for
// N(0, 1) keys) are rotated again from the float64 angle with float-float
// sin / cos (within 2^-46 (|a| + |b|)); only where even that leaves the
// rounding open is the float64 rotation itself computed.
//
// Error bound of the fp32 rotation (per element, |a|, |b| the bf16 inputs):
//   angle: the fractional turn pos * f_d / (2 pi) is exact modulo 2^64 in 0.64
//     fixed point; the turn constant carries at most |pos| 2^-51 rad against
//     the float64 product pos * f_d, which itself is rounded by |pos| 2^-53;
//   sin / cos: the top 24 bits of the turn go to sincospif exactly (its
//     documented error is 1 ulp, below 2^-24 for results of magnitude < 1;
//     2^-23 is assumed), the lower 40 bits (< 3.7e-7 rad) are added by the
//     first-order angle-sum correction (second-order term < 7e-14, correction
//     rounded within 2^-24);
//   so |cos - cos(phi)|, |sin - sin(phi)| <= delta = 3 * 2^-24 + |pos| 2^-50;
//   the rotation fmaf(a, c, -(b s)) adds |b s| 2^-24 + |y| 2^-24.
// E = (|a| + |b|) (delta + 2^-24) + |y| 2^-24, computed with a factor of
// safety (the 2^-22 terms below).
constexpr float kRopeSinCosErr = 3.0f * 0x1p-24f;

// bf16 bits of the float64 value y, rounded to nearest even without double
// rounding: the float64 -> fp32 step truncates and records in the last fp32
// bit whether anything was dropped (round to odd), so the fp32 -> bf16
// rounding sees every bit below the ones it keeps.
__device__ __forceinline__ uint32_t bf16_bits_rne(double y) {
  const float t = __double2float_rz(y);
  uint32_t u = __float_as_uint(t);
  if (static_cast<double>(t) != y) u |= 1u;
  return (u + 0x7fffu + ((u >> 16) & 1u)) >> 16;
}

__device__ __forceinline__ uint32_t bf16_bits_rn(float x) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  return static_cast<uint32_t>(*reinterpret_cast<const unsigned short*>(&h));
}

// Does every value within e of x round to the same bf16?
__device__ __forceinline__ bool bf16_rounding_decided(float x, float e) {
  return bf16_bits_rn(__fsub_rd(x, e)) == bf16_bits_rn(__fadd_ru(x, e));
}

// The rotated pair (a cos(phi) - b sin(phi), b cos(phi) + a sin(phi)) at
// phi = pos * freq in float64, in the definition's order of operations (phi
// rounded, each product rounded, then the difference / sum), each rounded to
// bf16: low 16 bits the first, high 16 bits the second.  Kept out of line: it
// runs only where the float-float rotation leaves the rounding open.
static __device__ __noinline__ uint32_t rope_pair_f64(int pos, double freq, float a, float b) {
  const double phi = __dmul_rn(static_cast<double>(pos), freq);
  double sd, cd;
  sincos(phi, &sd, &cd);
  const double ad = a, bd = b;
  const uint32_t ra = bf16_bits_rne(__dsub_rn(__dmul_rn(ad, cd), __dmul_rn(bd, sd)));
  const uint32_t rb = bf16_bits_rne(__dadd_rn(__dmul_rn(bd, cd), __dmul_rn(ad, sd)));
  return ra | (rb << 16);
}

// ---- second tier: the float64 angle, reduced exactly, and float-float sin / cos
//
// Float-float (hi + lo, two fp32 values) carries about 48 bits; float64 runs at
// a small fraction of the fp32 rate on this part, so the second tier uses one
// float64 instruction only -- the product phi = pos * f_d, rounded as the
// definition rounds it -- and does the rest in integer and fp32 arithmetic.
struct FF {
  float hi, lo;
};

// a * b exactly as hi + lo (fma-based two-product).
__device__ __forceinline__ FF ff_two_prod(float a, float b) {
  const float p = __fmul_rn(a, b);
  return {p, fmaf(a, b, -p)};
}

// a + b exactly as hi + lo (two-sum).
__device__ __forceinline__ FF ff_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  return {s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb))};
}

__device__ __forceinline__ FF ff_mul(FF x, FF y) {
  FF p = ff_two_prod(x.hi, y.hi);
  p.lo = fmaf(x.hi, y.lo, fmaf(x.lo, y.hi, p.lo));
  return ff_two_sum(p.hi, p.lo);
}

__device__ __forceinline__ FF ff_add(FF x, FF y) {
  FF s = ff_two_sum(x.hi, y.hi);
  s.lo = __fadd_rn(s.lo, __fadd_rn(x.lo, y.lo));
  return ff_two_sum(s.hi, s.lo);
}

__device__ __forceinline__ FF ff_neg(FF x) { return {-x.hi, -x.lo}; }

// phi / (2 pi) mod 1 as a 0.64 fixed-point fraction (two's complement for a
// negative phi), from the exact binary value of phi (m 2^(e - 1075)) and
// 1 / (2 pi) to 128 bits: floor(2^128 / (2 pi)) = 0x28be60db9391054a_7f09d5f47d4d3770
// (from pi by Machin's formula, 16 atan(1/5) - 4 atan(1/239), in integer
// arithmetic).  Exact up to the truncation of that constant, below 2^-90 turn
// for |phi| < 2^31.
__device__ __forceinline__ unsigned long long turn_fraction(double phi) {
  const unsigned long long bits = static_cast<unsigned long long>(__double_as_longlong(phi));
  const int ex = static_cast<int>((bits >> 52) & 0x7ffu);
  if (ex == 0) return 0;  // zero (a subnormal angle is below 1e-307 turn)
  const unsigned long long m = (bits & ((1ull << 52) - 1)) | (1ull << 52);
  constexpr unsigned long long kRh = 0x28be60db9391054aull, kRl = 0x7f09d5f47d4d3770ull;
  // m * R as 192 bits (p2, p1; the lowest limb is never needed)
  const unsigned long long h0 = __umul64hi(m, kRl);
  const unsigned long long l1 = m * kRh, h1 = __umul64hi(m, kRh);
  const unsigned long long p1 = h0 + l1;
  const unsigned long long p2 = h1 + (p1 < h0 ? 1ull : 0ull);
  const int sh = 1139 - ex;  // frac(phi / 2 pi) 2^64 = (m R) >> sh, mod 2^64
  unsigned long long f;
  if (sh >= 192) f = 0;
  else if (sh >= 128) f = p2 >> (sh - 128);
  else if (sh > 64) f = (p1 >> (sh - 64)) | (p2 << (128 - sh));
  else f = p1;  // sh >= 86 whenever |phi| < 2^31 (a 32-bit position times f_d <= 1)
  return (bits >> 63) ? 0ull - f : f;
}

// The rotated pair of rope_pair_f64, from the same float64 angle phi =
// pos * freq, with sin / cos in float-float: the turn fraction's top 8 bits
// pick cos / sin(2 pi k / 256) from kRopeTurnTable (float-float, within
// 2^-50), the remaining t < 2 pi / 256 rad goes through its Taylor
// series (sin: t - t^3/6 + t^5/120, cos: 1 - t^2/2 + t^4/24 - t^6/720; the
// first dropped terms are below 2^-49), and the angle sum combines them.
// Every value is within 2^-46 (|a| + |b|) of the float64 rotation; when the
// bf16 rounding is still open within that bound (an element within about one
// fp32 ulp of a rounding midpoint), *decided is false and the caller falls
// back to the float64 rotation.
__device__ uint32_t rope_pair_ff(int pos, double freq, float a, float b, float c_hi, float c_lo, bool* decided) {
  const unsigned long long f = turn_fraction(__dmul_rn(static_cast<double>(pos), freq));
  const int k = static_cast<int>(f >> 56);
  const unsigned long long r = f & ((1ull << 56) - 1);
  // t = 2 pi r / 2^64 = r (c_hi + c_lo) in float-float
  const float r_hi = static_cast<float>(static_cast<unsigned>(r >> 32)) * 0x1p32f;  // exact
  const float r_lo = static_cast<float>(static_cast<unsigned>(r & 0xffffffffull));
  FF t = ff_two_prod(r_hi, c_hi);
  t.lo = fmaf(r_hi, c_lo, fmaf(r_lo, c_hi, t.lo));
  t = ff_two_sum(t.hi, t.lo);
  FF t2 = ff_two_prod(t.hi, t.hi);
  t2.lo = fmaf(2.f * t.hi, t.lo, t2.lo);
  FF t3 = ff_two_prod(t2.hi, t.hi);
  t3.lo = fmaf(t2.hi, t.lo, fmaf(t2.lo, t.hi, t3.lo));
  // t^3 / 6: quotient rounded, exact remainder
  const float q = __fdiv_rn(t3.hi, 6.f);
  const float q_lo = __fdiv_rn(__fadd_rn(fmaf(-q, 6.f, t3.hi), t3.lo), 6.f);
  const float t4 = __fmul_rn(t2.hi, t2.hi);
  FF sn = ff_two_sum(t.hi, -q);
  sn.lo = __fadd_rn(sn.lo, __fsub_rn(t.lo, q_lo) + __fmul_rn(t4, t.hi) * (1.f / 120.f));
  FF cs = ff_two_sum(1.f, -0.5f * t2.hi);
  cs.lo = __fadd_rn(cs.lo, -0.5f * t2.lo + t4 * (1.f / 24.f) - __fmul_rn(t4, t2.hi) * (1.f / 720.f));
  sn = ff_two_sum(sn.hi, sn.lo);
  cs = ff_two_sum(cs.hi, cs.lo);
  const float4 kt = __ldg(reinterpret_cast<const float4*>(kRopeTurnTable) + k);
  const FF kc = {kt.x, kt.y};
  const FF ks = {kt.z, kt.w};
  const FF cphi = ff_add(ff_mul(kc, cs), ff_neg(ff_mul(ks, sn)));
  const FF sphi = ff_add(ff_mul(ks, cs), ff_mul(kc, sn));
  // y1 = a cos - b sin, y2 = b cos + a sin (a, b exact in fp32)
  const FF y1 = ff_add(ff_mul({a, 0.f}, cphi), ff_neg(ff_mul({b, 0.f}, sphi)));
  const FF y2 = ff_add(ff_mul({b, 0.f}, cphi), ff_mul({a, 0.f}, sphi));
  const float e = (fabsf(a) + fabsf(b)) * 0x1p-44f;
  uint32_t out = 0;
  bool ok = true;
  const FF ys[2] = {y1, y2};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    // y = hi + lo: its distance to m, the midpoint of hi's bf16 interval (hi - m
    // is exact: both share their top 16 bits), decides the rounding unless it is
    // within e; the neighbouring intervals' midpoints are 2^15 fp32 ulps away
    const uint32_t u = __float_as_uint(ys[i].hi);
    const float m = __uint_as_float((u & 0xffff0000u) | 0x8000u);
    const float d = __fadd_rn(__fsub_rn(ys[i].hi, m), ys[i].lo);
    ok = ok && fabsf(d) > e;
    // |y| above |m| rounds the magnitude up to the next bf16 value
    const bool up = (d > 0.f) == (ys[i].hi > 0.f);
    out |= ((u >> 16) + (up ? 1u : 0u)) << (16 * i);
  }
  *decided = ok;
  return out;
}

// cos / sin of 2 pi * (pos * turns mod 2^64) / 2^64 (the turn as a 0.64
// fixed-point fraction) in fp32, within kRopeSinCosErr of the exact values.
__device__ __forceinline__ void rope_cos_sin(int pos, unsigned long long turns, float& c, float& s) {
  const long long prod = static_cast<long long>(static_cast<unsigned long long>(static_cast<long long>(pos)) * turns);
  // top 24 bits: half-turns in [-1, 1), exact in fp32
  const float x_hi = static_cast<float>(static_cast<int>(prod >> 40)) * 0x1p-23f;
  // lower 40 bits: the rest of the angle, below 2 pi 2^-24 rad
  const float th_lo = static_cast<float>(static_cast<unsigned long long>(prod) & 0xffffffffffull) *
                      (6.283185307179586f * 0x1p-64f);
  float sh, ch;
  sincospif(x_hi, &sh, &ch);
  c = fmaf(-sh, th_lo, ch);
  s = fmaf(ch, th_lo, sh);
}

// The K/V tiles of one CTA: the shared prefix tiles, then the private tiles of
// every rollout its packed rows belong to.  Pure arithmetic, identical in every
// thread; split `split` of `num_splits` takes a contiguous share of the list.
struct TileRange {
  int lo, hi;       // [lo, hi) in the CTA's list
  int r_first;      // first rollout of the CTA's rows
  int n_priv;       // private tiles per rollout
};

__device__ __forceinline__ TileRange tile_range(const AttnParams& p, int m0, int split) {
  const int per_roll = p.n_q * p.G;
  const int row_end = min(m0 + BM, p.rows_per_head);
  TileRange tr;
  tr.r_first = m0 / per_roll;
  const int r_last = (row_end - 1) / per_roll;
  tr.n_priv = p.q_pos ? 0 : (p.priv_len + p.n_q + BN - 1) / BN;  // streaming mask: no own keys
  const int total = p.n_prefix_tiles + (r_last - tr.r_first + 1) * tr.n_priv;
  // ceil boundaries: when the splits cannot all take the same number of
  // tiles, the last split (which holds the diagonal tiles of the active
  // block, the slowest to process) is among those that take fewer
  tr.lo = static_cast<int>((static_cast<long long>(split) * total + p.num_splits - 1) / p.num_splits);
  tr.hi = static_cast<int>((static_cast<long long>(split + 1) * total + p.num_splits - 1) / p.num_splits);
  return tr;
}

__device__ __forceinline__ TileEntry tile_at(const AttnParams& p, const TileRange& tr, int t) {
  const int j = tr.lo + t;
  if (j < p.n_prefix_tiles) return {-1, j * BN};
  const int k = j - p.n_prefix_tiles;
  return {tr.r_first + k / tr.n_priv, (k % tr.n_priv) * BN};
}

// Merges the KV splits of a cluster (one CTA per split, same rows).  Called by
// every thread of every CTA of the cluster once its own K/V range is done:
//   1. each softmax thread writes its half of its row -- O / l in bf16 from
//      TMEM -- into the workspace slice of the CTA that owns the row, and its
//      (running max m, sum l) straight into that CTA's shared memory;
//   2. cluster barrier (release / acquire): every split's rows are written;
//   3. CTA q owns rows [q * r, (q + 1) * r): one thread pulls its S O slices
//      (contiguous) into shared memory with one bulk copy; meanwhile each
//      softmax thread takes a (row, 8 columns) item and forms its row's
//      weights l_s 2^(m_s - M) / L (M = max m_s, L = sum l_s 2^(m_s - M)),
//      then stores O = sum w_s O_s in bf16 and, for the first 8 columns,
//      LSE = (M + log2 L) ln 2.
template <int D, bool KV8>
__device__ void cluster_merge(const AttnParams& p, uint8_t* smem, uint32_t tmem, int m0, bool have_o, float m_run,
                              float l_tot, uint64_t* bars, volatile int* abort_flag) {
  using L = Layout<D, KV8>;
  constexpr int kCh = D / 8;  // bf16x8 chunks of a row
  constexpr int kThreads = 32 * kSmWarps;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool is_sm = warp >= 2 && warp < 2 + kSmWarps;
  const int S = p.num_splits;
  const int split = blockIdx.x;
  const int rpc = attn_merge_rows(S);
  int32_t* ds = p.dev_status;
  uint4* part_o = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.part) +
                                           (static_cast<size_t>(blockIdx.z) * p.m_tiles + p.m_tile0 + blockIdx.y) *
                                               attn_part_bytes(S, D));  // [owner][split][kCh][rpc]
  float2* recv_ml = reinterpret_cast<float2*>(smem + L::kMLRecv);         // [S][rpc]
  if (is_sm) {
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    const int rl = quad * 32 + lane;
    if (__any_sync(0xffffffffu, m0 + rl < p.rows_per_head)) {
      const int q = rl / rpc;
      const int r = rl - q * rpc;
      uint4* dst = part_o + static_cast<size_t>(q * S + split) * kCh * rpc + r;
      const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16) + 2 * BN + half * (D / 2);
      const float inv_l = have_o && l_tot > 0.f ? 1.f / l_tot : 0.f;
      float v[32];
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        if (have_o) {
          tmem_ld32(lane_base + c * 32, v);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = 0.f;
        }
#pragma unroll
        for (int q8 = 0; q8 < 4; ++q8)
          __stcg(dst + (half * (kCh / 2) + c * 4 + q8) * rpc,
                 make_uint4(pack_bf16x2(v[8 * q8 + 0] * inv_l, v[8 * q8 + 1] * inv_l),
                            pack_bf16x2(v[8 * q8 + 2] * inv_l, v[8 * q8 + 3] * inv_l),
                            pack_bf16x2(v[8 * q8 + 4] * inv_l, v[8 * q8 + 5] * inv_l),
                            pack_bf16x2(v[8 * q8 + 6] * inv_l, v[8 * q8 + 7] * inv_l)));
      }
      if (half == 0)
        st_cluster_v2(cluster_addr(smem_addr(recv_ml + split * rpc + r), q), m_run, have_o ? l_tot : 0.f);
      fence_proxy_async_global();
    }
  }
  cluster_arrive();  // release: this split's slices are written
  cluster_wait();    // acquire: every split's slices are written
  const int r0 = split * rpc;
  const int mine = max(0, min(min(BM - r0, rpc), p.rows_per_head - m0 - r0));
  if (mine == 0) return;
  uint4* recv_o = reinterpret_cast<uint4*>(smem + L::kRecv);  // [S][kCh][rpc]
  if (threadIdx.x == 0) {
    fence_proxy_async_global();
    mbar_arrive_expect_tx(&bars[MERGE_O], static_cast<uint32_t>(S * kCh * rpc * 16));
    // the S slices of this owner are contiguous: one copy (measured faster
    // than one copy per slice)
    bulk_load(recv_o, part_o + static_cast<size_t>(split * S) * kCh * rpc, S * kCh * rpc * 16, &bars[MERGE_O]);
    // the copies land before this thread reaches the CTA's final barrier
    mbar_drain(&bars[MERGE_O], 0, ds);
  }
  if (!is_sm) return;
  const int t = threadIdx.x - 64;
  const int per_roll = p.n_q * p.G;
  const int kvh = blockIdx.z;
  for (int it = t; it < mine * kCh; it += kThreads) {
    const int ch = it / mine;  // consecutive threads: consecutive rows of one chunk
    const int j = it - ch * mine;
    const int grow = m0 + r0 + j;
    const int r_row = grow / per_roll;
    const int rem = grow - r_row * per_roll;
    const int i_row = rem / p.G;
    const int qhead = kvh * p.G + (rem - i_row * p.G);
    const size_t orow = (static_cast<size_t>(r_row) * p.n_q + i_row) * p.Hq + qhead;
    // the splits' weights l_s 2^(m_s - M) for row j, while the slices are in
    // flight; every load is issued unconditionally (indices clamped to the S
    // splits, the surplus weighted 0) so that none waits for another
    float2 ml[kAttnMaxSplits];
#pragma unroll
    for (int s2 = 0; s2 < kAttnMaxSplits; ++s2) ml[s2] = recv_ml[min(s2, S - 1) * rpc + j];
    float M = -INFINITY;
#pragma unroll
    for (int s2 = 0; s2 < kAttnMaxSplits; ++s2)
      if (s2 < S && ml[s2].y > 0.f) M = fmaxf(M, ml[s2].x);
    float Ls = 0.f;
#pragma unroll
    for (int s2 = 0; s2 < kAttnMaxSplits; ++s2) {
      ml[s2].y = s2 < S && ml[s2].y > 0.f ? ml[s2].y * fast_exp2(ml[s2].x - M) : 0.f;
      Ls += ml[s2].y;
    }
    const float inv = Ls > 0.f ? fast_rcp(Ls) : 0.f;
    if (it == t && !mbar_wait(&bars[MERGE_O], 0, abort_flag, ds, p.wait_ns)) return;
    uint4 x[kAttnMaxSplits];
#pragma unroll
    for (int s2 = 0; s2 < kAttnMaxSplits; ++s2) x[s2] = recv_o[(min(s2, S - 1) * kCh + ch) * rpc + j];
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int s2 = 0; s2 < kAttnMaxSplits; ++s2) {
      const float w = ml[s2].y * inv;
      const uint32_t xw[4] = {x[s2].x, x[s2].y, x[s2].z, x[s2].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float a, b;
        bf16x2_unpack(xw[e], a, b);
        fma2(acc[2 * e], acc[2 * e + 1], w, w, a, b, acc[2 * e], acc[2 * e + 1]);
      }
    }
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + orow * D + ch * 8) =
        make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                   pack_bf16x2(acc[6], acc[7]));
    if (ch == 0 && p.lse)
      p.lse[(static_cast<size_t>(r_row) * p.Hq + qhead) * p.n_q + i_row] =
          Ls > 0.f ? (M + fast_log2(Ls)) * kLn2 : -INFINITY;
  }
}

// The n-th of the 2 nt E4M3 tiles of a CTA in the converters' order: K 0,
// then K(j + 1) (while j + 1 < nt) and V(j) for j = 0 .. nt - 1 -- the order in
// which the products need them (S(t + 1) is issued before P.V(t)).
__device__ __forceinline__ void kv8_item(int n, int nt, int& t, bool& is_v) {
  if (n == 0) {
    t = 0;
    is_v = false;
  } else if (n - 1 < 2 * (nt - 1)) {
    t = ((n - 1) >> 1) + (((n - 1) & 1) ? 0 : 1);
    is_v = ((n - 1) & 1) != 0;
  } else {
    t = nt - 1;
    is_v = true;
  }
}

// 2^e in fp16 (e in [-15, 7]: 2^-15 is subnormal), both halves.
__device__ __forceinline__ __half2 pow2_f16x2(int e) {
  const unsigned short b = e >= -14 ? static_cast<unsigned short>((15 + e) << 10) : static_cast<unsigned short>(0x0200);
  const __half h = __ushort_as_half(b);
  return __halves2half2(h, h);
}

// Sixteen E4M3 bytes to sixteen fp16 values times 2^e (exact: the products
// stay within fp16's range and grid for e in [-15, 7]).
__device__ __forceinline__ void e4m3x16_to_f16(uint4 x, __half2 sc, uint4& lo, uint4& hi) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  uint32_t r[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t a = e4m3x2_to_f16x2(static_cast<uint16_t>(w[i] & 0xffffu));
    const uint32_t b = e4m3x2_to_f16x2(static_cast<uint16_t>(w[i] >> 16));
    const __half2 ha = __hmul2(*reinterpret_cast<const __half2*>(&a), sc);
    const __half2 hb = __hmul2(*reinterpret_cast<const __half2*>(&b), sc);
    r[2 * i] = *reinterpret_cast<const uint32_t*>(&ha);
    r[2 * i + 1] = *reinterpret_cast<const uint32_t*>(&hb);
  }
  lo = make_uint4(r[0], r[1], r[2], r[3]);
  hi = make_uint4(r[4], r[5], r[6], r[7]);
}

// Two bf16 values to two fp16 values (exact for 2^-17 <= |x| < 65504).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  float lo, hi;
  bf16x2_unpack(w, lo, hi);
  return pack_f16x2(lo, hi);
}

// FP8 K/V converters (kConvThreads threads): the queries' tile from bf16 to
// fp16 in place once it has landed, then every E4M3 K / V tile from its
// staging stage into its fp16 stage -- the 128-byte-swizzled layout that TMA
// gives a bf16 tile, which the products read -- scaled by the exponent of
// each row's 128-row block.  Rows past the segment arrive as zero bytes (TMA
// fill) and stay zero.  An exponent outside [-15, 7] is clamped and
// BD_DEV_BAD_INPUT recorded.
template <int D, bool KV8>
__device__ void convert_kv8(const AttnParams& p, const TileRange& tr, int nt, uint8_t* smem, uint64_t* bars,
                            volatile int* abort_flag, int kvh) {
  using L = Layout<D, KV8>;
  constexpr int kKSt = L::kKSt;
  constexpr int kCPR = D / 16;        // 16-byte E4M3 chunks of a key row
  constexpr int kChunks = BN * kCPR;  // of a tile
  const int ct = static_cast<int>(threadIdx.x) - 32 * (2 + kSmWarps);
  int32_t* ds = p.dev_status;
  bool ok = mbar_wait(&bars[QFULL], 0, abort_flag, ds, p.wait_ns);
  if (ok) {
    uint4* q = reinterpret_cast<uint4*>(smem + L::kQ);
    for (int i = ct; i < L::kQBytes / 16; i += kConvThreads) {
      uint4 w = q[i];
      w = make_uint4(bf16x2_to_f16x2(w.x), bf16x2_to_f16x2(w.y), bf16x2_to_f16x2(w.z), bf16x2_to_f16x2(w.w));
      q[i] = w;
    }
    fence_proxy_async_smem();  // generic writes before the products read them
  }
  mbar_arrive(&bars[QCONV]);
  bool bad = false;
  for (int n = 0; ok && n < 2 * nt; ++n) {
    int t;
    bool is_v;
    kv8_item(n, nt, t, is_v);
    // the tile's exponents -- its 128 rows span at most two 128-row blocks --
    // are fetched before the waits, so that they have landed by then
    const TileEntry te = tile_at(p, tr, t);
    const int8_t* ex;
    int row0, valid, n_blk;
    if (te.rollout < 0) {
      ex = (is_v ? p.pv_exp : p.pk_exp) + static_cast<size_t>(kvh) * p.p_exp_stride;
      row0 = te.key0;
      valid = p.C - te.key0;
      n_blk = p.p_exp_stride;
    } else {
      ex = (is_v ? p.rv_exp : p.rk_exp) + (static_cast<size_t>(te.rollout) * p.Hkv + kvh) * p.r_exp_stride;
      row0 = p.r_exp_row0 + te.key0;
      valid = p.priv_len + p.n_q - te.key0;
      n_blk = p.r_exp_stride;
    }
    const int blk0 = row0 >> 7;
    const int split_row = (blk0 + 1) * 128 - row0;  // first row of the tile in the second block
    const bool two = (valid < BN ? valid : BN) > split_row && blk0 + 1 < n_blk;
    int e0 = __ldg(ex + blk0);
    int e1 = two ? __ldg(ex + blk0 + 1) : 0;
    if (e0 < -15 || e0 > 7 || e1 < -15 || e1 > 7) {
      bad = true;
      e0 = e0 < -15 ? -15 : (e0 > 7 ? 7 : e0);
      e1 = e1 < -15 ? -15 : (e1 > 7 ? 7 : e1);
    }
    const __half2 sc0 = pow2_f16x2(e0), sc1 = pow2_f16x2(e1);
    const int st = n % kStgStages;
    if (!mbar_wait(&bars[STG_FULL + st], (n / kStgStages) & 1, abort_flag, ds, p.wait_ns)) break;
    const int stages = is_v ? kVStages : kKSt;
    const int slot = t % stages;
    // the fp16 stage holds tile t - stages until its product is done
    if (t >= stages &&
        !mbar_wait(&bars[(is_v ? VEMPTY : KEMPTY) + slot], (t / stages - 1) & 1, abort_flag, ds, p.wait_ns))
      break;
    const uint8_t* stg = smem + L::kStg + st * L::kStgBytes;
    uint8_t* dst = smem + (is_v ? L::kV : L::kK) + slot * L::kKVBytes;
#pragma unroll 4
    for (int c = ct; c < kChunks; c += kConvThreads) {
      const int row = c / kCPR;
      const int col = (c - row * kCPR) * 16;
      const uint4 x = *reinterpret_cast<const uint4*>(stg + c * 16);
      // rows past the segment hold zero bytes: any scale keeps them zero
      uint4 lo, hi;
      e4m3x16_to_f16(x, row >= split_row ? sc1 : sc0, lo, hi);
      *reinterpret_cast<uint4*>(dst + sw128_offset(row, col, BN)) = lo;
      *reinterpret_cast<uint4*>(dst + sw128_offset(row, col + 8, BN)) = hi;
    }
    fence_proxy_async_smem();
    mbar_arrive(&bars[(is_v ? VFULL : KFULL) + slot]);
    mbar_arrive(&bars[STG_EMPTY + st]);
  }
  if (bad && ds) atomicOr(ds, BD_DEV_BAD_INPUT);
}

// STREAM: the streaming mask (q_pos), compiled apart so that the block-causal
// path carries none of its code.  KV8: E4M3 K/V with power-of-two block
// scales, dequantised to fp16 in shared memory by two more warps; the products
// then take fp16 operands (queries converted in place).
template <int D, bool STREAM, bool KV8>
__global__ void __launch_bounds__(threads_of<KV8>(), 1)
    attn_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ AttnMaps maps) {
  using L = Layout<D, KV8>;
  constexpr int kKSt = L::kKSt;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::kMisc);  // [0] tmem base, [1] abort
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int split = blockIdx.x;
  const int m0 = (p.m_tile0 + blockIdx.y) * BM;
  const int kvh = blockIdx.z;
  int32_t* ds = p.dev_status;

  const TileRange tr = tile_range(p, m0, split);
  const int nt = tr.hi - tr.lo;
  // TMA of K tile t into K stage t % 3 and of V tile t into V stage t % 2 (the
  // caller has made sure the stage is free)
  auto issue_tile = [&](int t, bool is_v) {
    const int s = is_v ? t % kVStages : t % kKSt;
    const TileEntry te = tile_at(p, tr, t);
    uint8_t* dst = smem + (is_v ? L::kV : L::kK) + s * L::kKVBytes;
    uint64_t* bar = &bars[(is_v ? VFULL : KFULL) + s];
    const CUtensorMap* pm = is_v ? &maps.pv : &maps.pk;
    const CUtensorMap* rm = is_v ? &maps.rv : &maps.rk;
    mbar_arrive_expect_tx(bar, L::kKVBytes);
#pragma unroll
    for (int hh = 0; hh < D / 64; ++hh) {
      if (te.rollout < 0)
        tma_load_3d(dst + hh * BN * 128, pm, hh * 64, te.key0, kvh, bar);
      else
        tma_load_4d(dst + hh * BN * 128, rm, hh * 64, te.key0, kvh, te.rollout, bar);
    }
  };

  // The first K/V loads (K 0, V 0, K 1, V 1, K 2 -- K runs one tile ahead of
  // V): with early = true only the leading prefix tiles among them, issued
  // before the dependency wait; with early = false the rest.
  // FP8 K/V: the n-th E4M3 tile in the converters' order (kv8_item) by TMA
  // into staging stage n % kStgStages (the caller has made sure the stage is
  // free)
  auto issue_item = [&](int n) {
    int t;
    bool is_v;
    kv8_item(n, nt, t, is_v);
    const TileEntry te = tile_at(p, tr, t);
    uint8_t* dst = smem + L::kStg + (n % kStgStages) * L::kStgBytes;
    uint64_t* bar = &bars[STG_FULL + n % kStgStages];
    mbar_arrive_expect_tx(bar, L::kStgBytes);
    if (te.rollout < 0)
      tma_load_3d(dst, is_v ? &maps.pv : &maps.pk, 0, te.key0, kvh, bar);
    else
      tma_load_4d(dst, is_v ? &maps.rv : &maps.rk, 0, te.key0, kvh, te.rollout, bar);
  };

  auto issue_initial = [&](bool early) {
    if constexpr (KV8) {
      if (!early)
        for (int n = 0; n < kStgStages && n < 2 * nt; ++n) issue_item(n);
    } else {
      for (int u = 0; u < 5; ++u) {
        const int t = u >> 1;
        const bool is_v = (u & 1) != 0;
        if (t >= nt) break;
        const bool prefix = tr.lo + t < p.n_prefix_tiles;
        if (early ? (prefix && p.prefix_early) : !(prefix && p.prefix_early)) issue_tile(t, is_v);
      }
    }
  };

  if (threadIdx.x == 0) {
    if (p.q_tma) tma_prefetch_desc(&maps.q);
    if (p.n_prefix_tiles > 0) {
      tma_prefetch_desc(&maps.pk);
      tma_prefetch_desc(&maps.pv);
    }
    tma_prefetch_desc(&maps.rk);
    tma_prefetch_desc(&maps.rv);
    // FP8 K/V: the fp16 stages are filled by the converter threads' arrivals
    for (int i = 0; i < kKSt; ++i) {
      mbar_init(&bars[KFULL + i], KV8 ? kConvThreads : 1);
      mbar_init(&bars[KEMPTY + i], 1);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(&bars[VFULL + i], KV8 ? kConvThreads : 1);
      mbar_init(&bars[VEMPTY + i], 1);
    }
    if (KV8) {
      mbar_init(&bars[QCONV], kConvThreads);
      for (int i = 0; i < kStgStages; ++i) {
        mbar_init(&bars[STG_FULL + i], 1);
        mbar_init(&bars[STG_EMPTY + i], kConvThreads);
      }
    }
    mbar_init(&bars[SFULL + 0], 1);
    mbar_init(&bars[SFULL + 1], 1);
    mbar_init(&bars[PFULL + 0], 32 * kSmWarps);
    mbar_init(&bars[PFULL + 1], 32 * kSmWarps);
    mbar_init(&bars[ODONE + 0], 1);
    mbar_init(&bars[ODONE + 1], 1);
    mbar_init(&bars[QFULL], p.q_tma ? 1 : 128);
    mbar_init(&bars[DRAIN], 1);
    mbar_init(&bars[MERGE_O], 1);
    misc[1] = 0;
    fence_mbar_init();
    // cached prefix tiles the caller declared complete before the previous
    // kernel of the stream started may be fetched before the dependency wait
    if (p.prefix_early) issue_initial(true);
  }
  if (warp == 1) {
    tmem_alloc(&misc[0], L::kTmemCols);
    tmem_relinquish();
  }
  // Everything above touches only shared memory, TMEM, the kernel's own
  // parameters and (prefix_early) cached prefix rows; from here on this thread
  // reads or writes global memory that the previous kernel in the stream may
  // still be producing.
  tc_fence_before();
  __syncthreads();  // barriers initialised, TMEM allocated
  tc_fence_after();
  pdl_wait();
  if (threadIdx.x == 0) {
    // the first loads leave as soon as this thread's wait returns
    if (nt > 0) {
      if (p.q_tma) {
        mbar_arrive_expect_tx(&bars[QFULL], L::kQBytes);
#pragma unroll
        for (int hh = 0; hh < D / 64; ++hh)
          tma_load_4d(smem + L::kQ + hh * BM * 128, &maps.q, hh * 64, 0, kvh, m0 / p.G, &bars[QFULL]);
      }
      issue_initial(false);
    }
  }
  pdl_trigger();  // the next kernel may start its own set-up on free SMs
  const uint32_t tmem = misc[0];
  // softmax state of this thread's packed row (softmax warps), kept for the merge
  float m_run = -INFINITY;  // running max, log2-scaled
  float l_run = 0.f;
  bool have_o = false;

  if (warp == 0 && KV8) {
    // ---------------------------------------------------------------- TMA producer (FP8 K/V)
    if (lane == 0 && nt > 0) {
      // item n goes into staging stage n % 3 once the converters are done with item n - 3
      int n = kStgStages < 2 * nt ? kStgStages : 2 * nt;  // items issued so far
      for (; n < 2 * nt; ++n) {
        if (!mbar_wait(&bars[STG_EMPTY + n % kStgStages], (n / kStgStages - 1) & 1, abort_flag, ds, p.wait_ns))
          break;
        issue_item(n);
      }
      if (p.q_tma) mbar_drain(&bars[QFULL], 0, ds);
      for (int u = n > kStgStages ? n - kStgStages : 0; u < n; ++u)
        mbar_drain(&bars[STG_FULL + u % kStgStages], (u / kStgStages) & 1, ds);
    }
  } else if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0 && nt > 0) {
      // K tile t + 1 needs S of tile t - 2 done (its stage), V tile t needs P.V
      // of tile t - 2 done; S(t - 2) completes before P.V(t - 3), so issuing in
      // the order K(t + 1), V(t) never waits behind a later event
      int nk = nt < 3 ? nt : 3, nv = nt < 2 ? nt : 2;  // tiles issued so far
      for (int t = 2; t < nt; ++t) {
        if (t + 1 < nt) {
          if (!mbar_wait(&bars[KEMPTY + (t + 1) % kKSt], ((t + 1) / kKSt - 1) & 1, abort_flag, ds, p.wait_ns)) break;
          issue_tile(t + 1, false);
          nk = t + 2;
        }
        if (!mbar_wait(&bars[VEMPTY + t % kVStages], (t / kVStages - 1) & 1, abort_flag, ds, p.wait_ns)) break;
        issue_tile(t, true);
        nv = t + 1;
      }
      // every copy issued lands before the CTA gives up its shared memory
      if (p.q_tma) mbar_drain(&bars[QFULL], 0, ds);
      for (int u = nk > kKSt ? nk - kKSt : 0; u < nk; ++u)
        mbar_drain(&bars[KFULL + u % kKSt], (u / kKSt) & 1, ds);
      for (int u = nv > kVStages ? nv - kVStages : 0; u < nv; ++u)
        mbar_drain(&bars[VFULL + u % kVStages], (u / kVStages) & 1, ds);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0 && nt > 0) {
      constexpr uint32_t kIdS = mma_idesc_16(BM, BN, false, !KV8);
      constexpr uint32_t kIdPV = mma_idesc_16(BM, D, true, !KV8);
      const uint32_t qa = smem_addr(smem + L::kQ);
      auto issue_s = [&](int u) -> bool {
        const int s = u & 1;
        const int ks = u % kKSt;
        // S buffer s held P(u - 2), which P.V(u - 2) -- issued before this
        // point by this thread, and executed in issue order -- has consumed
        if (!mbar_wait(&bars[KFULL + ks], (u / kKSt) & 1, abort_flag, ds, p.wait_ns)) return false;
        tc_fence_after();
        const uint32_t ka = smem_addr(smem + L::kK + ks * L::kKVBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t qoff = (kk >> 2) * (BM * 128) + (kk & 3) * 32;
          const uint32_t koff = (kk >> 2) * (BN * 128) + (kk & 3) * 32;
          mma_bf16(tmem + s * BN, sw128_desc(qa + qoff, 16, 1024), sw128_desc(ka + koff, 16, 1024), kIdS,
                   kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars[SFULL + s]);
        mma_commit(&bars[KEMPTY + ks]);  // K tile consumed: the producer may refill the stage
        return true;
      };
      // FP8 K/V: the queries once the converters have made them fp16
      bool ok = mbar_wait(&bars[KV8 ? QCONV : QFULL], 0, abort_flag, ds, p.wait_ns);
      if (ok) {
        tc_fence_after();
        ok = issue_s(0);
      }
      for (int t = 0; ok && t < nt; ++t) {
        if (t + 1 < nt && !issue_s(t + 1)) break;
        if (!mbar_wait(&bars[PFULL + (t & 1)], (t >> 1) & 1, abort_flag, ds, p.wait_ns)) break;
        if (!mbar_wait(&bars[VFULL + t % kVStages], (t / kVStages) & 1, abort_flag, ds, p.wait_ns)) break;
        tc_fence_after();
        const uint32_t va = smem_addr(smem + L::kV + (t % kVStages) * L::kKVBytes);
        const uint32_t pt = tmem + (t & 1) * BN;  // P(t), in the S buffer it was formed from
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          // keys [16 kk, 16 kk + 16): the half of the row that holds them, 8 packed columns
          const uint32_t acol = (kk >> 2) * (BN / 2) + (kk & 3) * 8;
          const uint32_t voff = kk * 16 * 128;
          mma_bf16_ts(tmem + 2 * BN, pt + acol, sw128_desc(va + voff, BN * 128, 1024), kIdPV,
                      (t > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&bars[ODONE + (t & 1)]);
        mma_commit(&bars[VEMPTY + t % kVStages]);
      }
      mma_commit(&bars[DRAIN]);
      mbar_drain(&bars[DRAIN], 0, ds);
    }
  } else if (KV8 && warp >= 2 + kSmWarps) {
    // ---------------------------------------------------------------- FP8 converters
    if (nt > 0) convert_kv8<D, KV8>(p, tr, nt, smem, bars, abort_flag, kvh);
  } else if (warp < 2 + kSmWarps) {
    // ---------------------------------------------------------------- softmax rows
    // Two warps per TMEM lane quadrant: warp 2 + 4h + q holds the rows of lanes
    // [32q, 32q + 32) and key columns [h BN/2, (h+1) BN/2) of each S tile (and
    // O columns [h D/2, (h+1) D/2)); the halves of a row trade their tile maxima
    // through shared memory and add their sums at the end.
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    const int rl = quad * 32 + lane;  // TMEM lane = packed row within the tile
    const int c0 = half * (BN / 2);   // first key column of this half
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
    if (!p.q_tma && half == 0) {  // GQA group that does not divide 128: rows gathered by the threads
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.q) + orow * D);
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const uint4 val = valid ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(smem + L::kQ + sw128_offset(rl, c * 8, BM)) = val;
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars[QFULL]);
    }

    const int lim_priv = valid && !STREAM ? p.priv_len + block_end_of(p, i_row) : 0;
    // streaming mask: this row's query position (nothing is visible to a padding row)
    const int qpos_row = valid && STREAM ? __ldg(p.q_pos + i_row) : INT_MIN;
    const bool warp_active = __any_sync(0xffffffffu, valid);
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    float* xch = reinterpret_cast<float*>(smem + L::kXch);
    bool ok = true;
    float v[32];
    // Named barrier 2 + quad is reached by the quadrant's two warps the same
    // number of times (nt + 1), whatever the waits return.
    for (int t = 0; t < nt; ++t) {
      const int s = t & 1;
      if (ok) ok = all_lanes(mbar_wait(&bars[SFULL + s], (t >> 1) & 1, abort_flag, ds, p.wait_ns));
      // this half of the S row in registers: one TMEM round trip, then S is free again
      float sv[BN / 2];
      float mx = -INFINITY;
      int nv = 0;
      bool dead = false;  // streaming mask: no row of this warp sees a key of this half tile
      if (ok) {
        tc_fence_after();
        const TileEntry te = tile_at(p, tr, t);
        int lim = te.rollout < 0 ? p.C : (te.rollout == r_row ? lim_priv : 0);
        if (!valid) lim = 0;
        nv = max(0, min(BN, lim - te.key0));
        if (warp_active) {
          if constexpr (STREAM) {
            // key j is visible iff its re-based position is at most the query's.
            // The range of the positions of this half tile (one 8-byte load per
            // lane, warp shuffles) settles most rows at once: every key visible
            // (nothing to mask) or none (the whole half masked); only when some
            // row's position falls inside the range are the keys compared one
            // by one, their positions read 16 bytes at a time
            const int kb = te.key0 + c0;
            const long long lim_q = static_cast<long long>(qpos_row) + p.kdelta;  // stored positions <= lim_q
            int kp_lo, kp_hi;
            if (p.kpos == nullptr) {
              kp_lo = kb;
              kp_hi = min(kb + BN / 2, p.C) - 1;
            } else {
              kp_lo = INT_MAX;
              kp_hi = INT_MIN;
              const int k2 = kb + 2 * lane;
              if (k2 + 1 < p.C) {
                const int2 kv = __ldg(reinterpret_cast<const int2*>(p.kpos + k2));
                kp_lo = min(kv.x, kv.y);
                kp_hi = max(kv.x, kv.y);
              } else if (k2 < p.C) {
                kp_lo = kp_hi = __ldg(p.kpos + k2);
              }
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) {
                kp_lo = min(kp_lo, __shfl_xor_sync(0xffffffffu, kp_lo, o));
                kp_hi = max(kp_hi, __shfl_xor_sync(0xffffffffu, kp_hi, o));
              }
            }
            const bool all_vis = kb + BN / 2 <= p.C && static_cast<long long>(kp_hi) <= lim_q;
            const bool none_vis = static_cast<long long>(kp_lo) > lim_q;
            dead = __all_sync(0xffffffffu, none_vis);  // S is then not even loaded
            if (!dead) tmem_ld64(lane_base + s * BN + c0, sv);
            if (!dead && !__all_sync(0xffffffffu, all_vis)) {
#pragma unroll
              for (int b = 0; b < BN / 64; ++b) {
                const int k0 = kb + 32 * b;
                if (p.kpos != nullptr && k0 + 32 <= p.C) {
                  int4 kp4[8];
#pragma unroll
                  for (int j4 = 0; j4 < 8; ++j4) kp4[j4] = __ldg(reinterpret_cast<const int4*>(p.kpos + k0) + j4);
#pragma unroll
                  for (int j4 = 0; j4 < 8; ++j4) {
                    if (kp4[j4].x > lim_q) sv[32 * b + 4 * j4 + 0] = -INFINITY;
                    if (kp4[j4].y > lim_q) sv[32 * b + 4 * j4 + 1] = -INFINITY;
                    if (kp4[j4].z > lim_q) sv[32 * b + 4 * j4 + 2] = -INFINITY;
                    if (kp4[j4].w > lim_q) sv[32 * b + 4 * j4 + 3] = -INFINITY;
                  }
                } else {
#pragma unroll
                  for (int j = 0; j < 32; ++j) {
                    const int key = k0 + j;
                    const int kp = key < p.C ? (p.kpos ? __ldg(p.kpos + key) : key) : INT_MAX;
                    if (key >= p.C || kp > lim_q) sv[32 * b + j] = -INFINITY;
                  }
                }
              }
            }
          } else {
            tmem_ld64(lane_base + s * BN + c0, sv);
            if (!__all_sync(0xffffffffu, nv >= c0 + BN / 2)) {
#pragma unroll
              for (int j = 0; j < BN / 2; ++j)
                if (c0 + j >= nv) sv[j] = -INFINITY;  // out of the max; exp2 gives 0
            }
          }
          if (!dead) {
            // eight independent chains of three-input maxima
            float m8[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) m8[q] = sv[q];
#pragma unroll
            for (int j = 8; j < BN / 2; j += 2) m8[(j >> 1) & 7] = fmax3(m8[(j >> 1) & 7], sv[j], sv[j + 1]);
            mx = fmaxf(fmax3(m8[0], m8[1], m8[2]), fmax3(fmax3(m8[3], m8[4], m8[5]), m8[6], m8[7]));
          }
        }
      }
      xch[(s * 2 + half) * BM + rl] = mx;
      named_sync(2 + quad, 64);  // the two halves of these 32 rows
      mx = fmaxf(mx, xch[(s * 2 + (half ^ 1)) * BM + rl]);
      if (!ok) continue;
      const float m_tile = nv > 0 ? mx * p.scale_log2 : -INFINITY;
      // both halves see the same m_tile and m_run, so they take the same decision
      const bool grow = m_tile > -INFINITY && (m_run == -INFINITY || m_tile > m_run + kRescaleLog2);
      float alpha = 1.f;
      if (grow) {
        alpha = (m_run == -INFINITY) ? 0.f : fast_exp2(m_run - m_tile);
        m_run = m_tile;
        l_run *= alpha;
      }
      // O must be rescaled (rare once the running max has settled): that needs
      // the previous tile's P.V to have finished first
      const bool rescale = warp_active && t > 0 && __any_sync(0xffffffffu, alpha != 1.f);
      if (rescale) {  // P.V(t - 1) must have finished updating O
        ok = all_lanes(mbar_wait(&bars[ODONE + ((t - 1) & 1)], ((t - 1) >> 1) & 1, abort_flag, ds, p.wait_ns));
        if (!ok) continue;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          const uint32_t oa = lane_base + 2 * BN + half * (D / 2) + c * 32;
          tmem_ld32(oa, v);
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] *= alpha;
          tmem_st32(oa, v);
        }
      }
      // P of this tile, rounded to bf16, goes into the first half of this
      // half's S columns (S buffer s), while the previous tile's P.V -- which
      // reads the other buffer -- is still running on the tensor pipe
      if (warp_active && dead) {
        // the half tile is hidden from every row of this warp: P = 0
        uint32_t zero[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) zero[j] = 0u;
#pragma unroll
        for (int c = 0; c < BN / 64; ++c) tmem_st16(lane_base + s * BN + c0 + 16 * c, zero);
        tmem_wait_st();
      } else if (warp_active) {
        // masked entries are -inf; a row that has seen no key yet keeps m_run = -inf
        const float mneg = m_run == -INFINITY ? 0.f : -m_run;
        float ls[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < BN / 64; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            float xa, xb;
            fma2(xa, xb, sv[32 * c + 2 * j], sv[32 * c + 2 * j + 1], p.scale_log2, p.scale_log2, mneg, mneg);
            const float a = fast_exp2(xa);
            const float b = fast_exp2(xb);
            add2(ls[2 * (j & 3)], ls[2 * (j & 3) + 1], a, b);
            pk[j] = KV8 ? pack_f16x2(a, b) : pack_bf16x2(a, b);
          }
          tmem_st16(lane_base + s * BN + c0 + 16 * c, pk);
        }
        l_run += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
        tmem_wait_st();
      }
      // P(t) does not wait for P.V(t - 1): it goes into the other S buffer.
      // The wait on P.V(t - 2) -- already done, since S(t) was issued after it
      // and tcgen05.mma runs in issue order -- only keeps this thread's view of
      // each ODONE barrier within one phase (no parity aliasing later).
      if (t >= 2) {
        ok = all_lanes(mbar_wait(&bars[ODONE + (t & 1)], ((t - 2) >> 1) & 1, abort_flag, ds, p.wait_ns));
        if (!ok) continue;
      }
      tc_fence_before();
      mbar_arrive(&bars[PFULL + (t & 1)]);
    }
    if (ok && nt > 0) {  // the last P.V (and, in issue order, every earlier one)
      ok = all_lanes(mbar_wait(&bars[ODONE + ((nt - 1) & 1)], ((nt - 1) >> 1) & 1, abort_flag, ds, p.wait_ns));
      tc_fence_after();
    }
    have_o = ok && nt > 0;
    xch[(4 + half) * BM + rl] = l_run;
    named_sync(2 + quad, 64);
    l_run += xch[(4 + (half ^ 1)) * BM + rl];  // the row's sum over both halves
    if (p.num_splits == 1) {
      const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
      if (warp_active) {
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          const int col = half * (D / 2) + c * 32;
          if (have_o) {
            tmem_ld32(lane_base + 2 * BN + col, v);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = 0.f;
          }
          if (!valid) continue;
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + orow * D + col);
#pragma unroll
          for (int qq = 0; qq < 4; ++qq)
            dst[qq] = make_uint4(pack_bf16x2(v[8 * qq + 0] * inv_l, v[8 * qq + 1] * inv_l),
                                 pack_bf16x2(v[8 * qq + 2] * inv_l, v[8 * qq + 3] * inv_l),
                                 pack_bf16x2(v[8 * qq + 4] * inv_l, v[8 * qq + 5] * inv_l),
                                 pack_bf16x2(v[8 * qq + 6] * inv_l, v[8 * qq + 7] * inv_l));
        }
      }
      if (valid && half == 0 && p.lse)
        p.lse[(static_cast<size_t>(r_row) * p.Hq + qhead) * p.n_q + i_row] =
            l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
    }
  }

  if (p.num_splits > 1) cluster_merge<D, KV8>(p, smem, tmem, m0, have_o, m_run, l_run, bars, abort_flag);

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

template <int D, bool STREAM, bool KV8>
cudaError_t launch_attn_t(AttnParams p, const AttnMaps& maps, int m_tiles, cudaStream_t stream) {
  static PerDeviceOnce configured;  // one per instantiation
  const int smem = attn_smem_bytes(D, KV8);
  auto kernel = attn_kernel<D, STREAM, KV8>;
  cudaError_t ce = configured.run([&] {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
  });
  if (ce != cudaSuccess) return ce;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  cfg.blockDim = dim3(threads_of<KV8>());
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  for (;;) {
    cfg.gridDim = dim3(p.num_splits, m_tiles, p.Hkv);
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = p.num_splits;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (p.num_splits <= 8) break;
    // a cluster wider than the portable 8 needs that many SMs free in one GPC
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) == cudaSuccess && n > 0) break;
    (void)cudaGetLastError();
    p.num_splits = 8;
  }
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, p, maps);
  return e == cudaSuccess ? cudaGetLastError() : e;
}

// Rotates the cached prefix keys [0, C) of every KV head at k_pos - delta into
// a contiguous bf16 copy [Hkv, C, D] (FlashDrive tutorial, "流式推理": the cache
// stays pre-RoPE; the operator applies the rotation at the re-based
// positions).  One thread per (KV head, key, 4 rotation pairs): the pairs
// (d, d + D/2) for d in [4 c, 4 c + 4).  Each rotated element is the bf16
// rounding (to nearest even) of the rotation computed in float64; see the
// error bound above.  The pairs whose rounding the fp32 rotation leaves open
// are queued in shared memory and redone, one pair per lane of whole warps,
// after the CTA's fast results are stored: from the float64 angle with
// float-float sin / cos, and in float64 where that still leaves the rounding
// open (float64 runs at a small fraction of the fp32 rate on this part).
constexpr int kRopeThreads = 256;
constexpr int kRopePairs = 4;     // rotation pairs (d, d + D/2) of one thread
constexpr int kRopeQueue = 512;   // queued pairs per CTA (a thread past it redoes its own)

struct RopeRedo {
  int pos;      // k_pos - delta
  int d;        // frequency index
  float a, b;   // the pair's pre-RoPE elements
  uint32_t at;  // element offset of the first output in the rotated copy
};

template <int D>
__global__ void __launch_bounds__(kRopeThreads) rope_prefix_kernel(const __grid_constant__ RopeParams p) {
  constexpr int kChunks = D / 2 / kRopePairs;  // chunks of kRopePairs pairs in a key row
  constexpr int kW = kRopePairs / 2;           // 32-bit words of a chunk's kRopePairs bf16 values
  using Vec = typename std::conditional<kW == 4, uint4, uint2>::type;
  __shared__ RopeRedo queue[kRopeQueue];
  __shared__ unsigned long long turns[D / 2];  // per-thread frequency indices vary within a warp: not from
  __shared__ int n_queued;                     // the constant bank, which serialises distinct addresses
  if (threadIdx.x == 0) n_queued = 0;
  for (int d = threadIdx.x; d < D / 2; d += blockDim.x) turns[d] = p.turns[d];
  pdl_wait();
  pdl_trigger();
  __syncthreads();
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long total = static_cast<long long>(p.Hkv) * p.C * kChunks;
  __nv_bfloat16* const out = static_cast<__nv_bfloat16*>(p.out);
  if (i < total) {
    const int c = static_cast<int>(i % kChunks);
    const long long row = i / kChunks;  // kvh * C + key
    const int key = static_cast<int>(row % p.C);
    const int kvh = static_cast<int>(row / p.C);
    const __nv_bfloat16* src =
        static_cast<const __nv_bfloat16*>(p.k) + (static_cast<size_t>(kvh) * p.stride + key) * D;
    __nv_bfloat16* dst = out + static_cast<size_t>(row) * D;
    const int pos = (p.k_pos ? __ldg(p.k_pos + key) : key) - p.delta;
    const float delta = kRopeSinCosErr + 0x1p-24f + static_cast<float>(abs(pos)) * 0x1p-50f;
    const int d0 = c * kRopePairs;
    Vec xa = __ldg(reinterpret_cast<const Vec*>(src + d0));
    Vec xb = __ldg(reinterpret_cast<const Vec*>(src + d0 + D / 2));
    const uint32_t* wa = reinterpret_cast<const uint32_t*>(&xa);
    const uint32_t* wb = reinterpret_cast<const uint32_t*>(&xb);
    float a[kRopePairs], b[kRopePairs], ya[kRopePairs], yb[kRopePairs];
#pragma unroll
    for (int w = 0; w < kW; ++w) {
      bf16x2_unpack(wa[w], a[2 * w], a[2 * w + 1]);
      bf16x2_unpack(wb[w], b[2 * w], b[2 * w + 1]);
    }
    unsigned redo = 0;  // pairs whose rounding the fp32 rotation does not settle
#pragma unroll
    for (int j = 0; j < kRopePairs; ++j) {
      float cs, sn;
      rope_cos_sin(pos, turns[d0 + j], cs, sn);
      ya[j] = fmaf(a[j], cs, -(b[j] * sn));
      yb[j] = fmaf(b[j], cs, a[j] * sn);
      const float e0 = (fabsf(a[j]) + fabsf(b[j])) * delta * (1.f + 0x1p-20f);
      const float ea = fmaf(fabsf(ya[j]), 0x1p-22f, e0);
      const float eb = fmaf(fabsf(yb[j]), 0x1p-22f, e0);
      if (!bf16_rounding_decided(ya[j], ea) || !bf16_rounding_decided(yb[j], eb)) redo |= 1u << j;
    }
    Vec oa, ob;
    uint32_t* pa = reinterpret_cast<uint32_t*>(&oa);
    uint32_t* pb = reinterpret_cast<uint32_t*>(&ob);
#pragma unroll
    for (int w = 0; w < kW; ++w) {
      pa[w] = pack_bf16x2(ya[2 * w], ya[2 * w + 1]);
      pb[w] = pack_bf16x2(yb[2 * w], yb[2 * w + 1]);
    }
    *reinterpret_cast<Vec*>(dst + d0) = oa;
    *reinterpret_cast<Vec*>(dst + d0 + D / 2) = ob;
    if (redo) {
      const uint32_t at = static_cast<uint32_t>(row * D + d0);
#pragma unroll
      for (int j = 0; j < kRopePairs; ++j) {
        if (!((redo >> j) & 1u)) continue;
        const int q = atomicAdd(&n_queued, 1);
        if (q < kRopeQueue) {
          queue[q] = RopeRedo{pos, d0 + j, a[j], b[j], at + j};
        } else {  // the queue is full (never with N(0, 1) keys): this thread redoes the pair itself
          const uint32_t r = rope_pair_f64(pos, p.freq[d0 + j], a[j], b[j]);
          reinterpret_cast<unsigned short*>(out)[at + j] = static_cast<unsigned short>(r & 0xffffu);
          reinterpret_cast<unsigned short*>(out)[at + j + D / 2] = static_cast<unsigned short>(r >> 16);
        }
      }
    }
  }
  // the fast results above are stored before the redone elements overwrite them
  __syncthreads();
  const int n = min(n_queued, kRopeQueue);
  for (int q = threadIdx.x; q < n; q += blockDim.x) {
    const RopeRedo it = queue[q];
    bool decided;
    uint32_t r = rope_pair_ff(it.pos, p.freq[it.d], it.a, it.b, p.two_pi_64[0], p.two_pi_64[1], &decided);
    if (!decided) r = rope_pair_f64(it.pos, p.freq[it.d], it.a, it.b);
    reinterpret_cast<unsigned short*>(out)[it.at] = static_cast<unsigned short>(r & 0xffffu);
    reinterpret_cast<unsigned short*>(out)[it.at + D / 2] = static_cast<unsigned short>(r >> 16);
  }
}

template <int D>
cudaError_t launch_rope_t(const RopeParams& p, cudaStream_t stream) {
  const long long total = static_cast<long long>(p.Hkv) * p.C * (D / 2 / kRopePairs);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(static_cast<unsigned>((total + kRopeThreads - 1) / kRopeThreads));
  cfg.blockDim = dim3(kRopeThreads);
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, rope_prefix_kernel<D>, p);
  return e == cudaSuccess ? cudaGetLastError() : e;
}

}  // namespace

int attn_smem_bytes(int D, bool kv8) {
  // D = 64 is padded so that one CTA (and its 512 TMEM columns) fills an SM.
  const int a = D == 128 ? (kv8 ? Layout<128, true>::kAlloc : Layout<128>::kAlloc)
                         : (kv8 ? Layout<64, true>::kAlloc : Layout<64>::kAlloc);
  return D == 128 || a > 120 * 1024 ? a : 120 * 1024;
}

int attn_max_clusters(int S, int D) {
  if (S < 1 || S > kAttnMaxSplits) return 0;
  static std::mutex mu;
  static int cache[64][2][kAttnMaxSplits + 1];  // 0: not asked yet, -1: no answer
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    (void)cudaGetLastError();
    return attn_resident_clusters(S);
  }
  std::lock_guard<std::mutex> lk(mu);
  int& c = cache[dev][D == 128 ? 1 : 0][S];
  if (c == 0) {
    auto kernel = D == 128 ? attn_kernel<128, false, false> : attn_kernel<64, false, false>;
    const int smem = attn_smem_bytes(D, false);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(S, 1, 1);
    cfg.blockDim = dim3(threads_of<false>());
    cfg.dynamicSmemBytes = smem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess &&
        cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess &&
        cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) == cudaSuccess) {
      c = n;
    } else {
      (void)cudaGetLastError();
      c = -1;
    }
  }
  return c >= 0 ? c : attn_resident_clusters(S);
}

cudaError_t launch_attention(const AttnParams& p, const AttnMaps& maps, int m_tiles, cudaStream_t stream) {
  if (p.q_pos)
    return p.D == 128 ? launch_attn_t<128, true, false>(p, maps, m_tiles, stream)
                      : launch_attn_t<64, true, false>(p, maps, m_tiles, stream);
  if (p.kv8)
    return p.D == 128 ? launch_attn_t<128, false, true>(p, maps, m_tiles, stream)
                      : launch_attn_t<64, false, true>(p, maps, m_tiles, stream);
  return p.D == 128 ? launch_attn_t<128, false, false>(p, maps, m_tiles, stream)
                    : launch_attn_t<64, false, false>(p, maps, m_tiles, stream);
}

cudaError_t launch_rope_prefix(const RopeParams& p, cudaStream_t stream) {
  if (p.Hkv < 1 || p.C < 1) return cudaSuccess;
  return p.D == 128 ? launch_rope_t<128>(p, stream) : launch_rope_t<64>(p, stream);
}

}  // namespace bd
