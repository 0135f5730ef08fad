// api.cu -- the extern "C" entry points of libbd (declared in include/bd.h):
// argument validation on the host, workspace sizing and carving, TMA tensor
// maps (cuTensorMapEncodeTiled through the runtime's driver entry point, so the
// library does not link libcuda), and the kernel launches of attn.cu / vocab.cu.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/bd.h"
#include "launch.h"

namespace {

using namespace bd;

// SMs of the current device, asked once per device; 152 (a full GB300) when
// no device answers, so that workspace sizes can be computed on a host without
// a GPU.  Plans -- and so workspace sizes -- are made for the current device.
int plan_sms() {
  static std::mutex mu;
  static int sms[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    (void)cudaGetLastError();
    return 152;
  }
  std::lock_guard<std::mutex> lk(mu);
  if (sms[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) {
      (void)cudaGetLastError();
      n = 152;
    }
    sms[dev] = n;
  }
  return sms[dev];
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Limit of a kernel's pipeline waits: the call's, or 1 s.
unsigned long long wait_limit(uint64_t ns) { return ns ? ns : 1000ull * 1000ull * 1000ull; }

// ------------------------------------------------------------------ device checks

std::mutex g_mu;
int g_dev_cc[64];  // 0 unknown, else major*10+minor

bd_status check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BD_ERR_CUDA;
  if (dev < 0 || dev >= 64) return BD_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_dev_cc[dev] == 0) {
    int ma = 0, mi = 0;
    if (cudaDeviceGetAttribute(&ma, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&mi, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return BD_ERR_CUDA;
    g_dev_cc[dev] = ma * 10 + mi;
  }
  return g_dev_cc[dev] == 103 ? BD_OK : BD_ERR_UNSUPPORTED;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// bf16 tensor map with 128-byte swizzle; the box is {64, 128, 1, ...} unless
// given.  With bytes = true: 8-bit elements, no swizzle, box {dims[0], 128, 1, ...}.
bd_status make_kv_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
                      const uint32_t* box_in = nullptr, bool bytes = false) {
  auto fn = encode_fn();
  if (!fn) return BD_ERR_CUDA;
  cuuint64_t gdim[4];
  cuuint64_t gstr[3];
  cuuint32_t box[4] = {bytes ? static_cast<cuuint32_t>(dims[0]) : 64u, static_cast<cuuint32_t>(kAttnBN), 1, 1};
  if (box_in)
    for (int i = 0; i < rank; ++i) box[i] = box_in[i];
  cuuint32_t estr[4] = {1, 1, 1, 1};
  for (int i = 0; i < rank; ++i) gdim[i] = dims[i];
  for (int i = 0; i < rank - 1; ++i) gstr[i] = strides[i];
  const CUresult r = fn(m, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank,
                        const_cast<void*>(base), gdim, gstr, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        bytes ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? BD_OK : BD_ERR_CUDA;
}

// ------------------------------------------------------------------ attention (plain and fork)

struct AttnDesc {
  int N;
  const void* q;
  const void* pk;
  const void* pv;
  long long prefix_stride;
  const void* rk;
  const void* rv;
  long long priv_stride;
  int priv_len;
  void* o;
  float* lse;
  const int32_t* block_start;
  int n_blocks, block_size, C, n_q, Hq, Hkv, D;
  float sm_scale;
  bd_rope rope;
  int num_splits;
  void* ws;
  size_t ws_bytes;
  int32_t* ds;
  int prefix_ready;
  const int32_t* q_pos;  // streaming mask (plain attention only)
  uint64_t wait_ns;
  int kv_dtype;          // 0 / BD_BF16 or BD_E4M3
  const int8_t *pk_exp, *pv_exp, *rk_exp, *rv_exp;
  int p_exp_stride, r_exp_stride, r_exp_row0;
};

// One call runs as one launch, or as two when its (row tile, KV head) groups
// exceed one wave of SMs: a bulk launch of whole waves with one CTA per group,
// then the remaining groups split wide across the SMs (instead of a second,
// nearly empty wave of unsplit groups).
struct AttnPart {
  int m_tile0, m_tiles, splits;
};

struct AttnPlan {
  int G, rows_per_head, m_tiles, n_prefix_tiles, splits;  // splits: widest over the parts
  int n_parts;
  AttnPart part[2];
  size_t rope_off;  // workspace offset of the rotated prefix keys (RoPE)
  size_t ws_bytes;
};

// KV split count for a launch of `groups` clusters (one per (row tile, KV
// head)) whose K/V lists hold up to T tiles of head dim D.  Among the S whose
// CTAs fit the SMs and whose clusters are all resident at once (one wave), the
// cheapest by a small model in units of one tile's softmax period, fitted to
// split sweeps of the workloads' shapes on GB300 (the widest on ties):
//   * ceil(T / S) tiles on the longest split;
//   * 1.5 for the cluster merge itself (S > 1), plus 0.7 for each extra pass
//     of its 256 threads over the r(S) rows x D / 8 chunks an owner merges;
//   * 0.3 when the split holding the last tile (the active block's diagonal
//     tile, the slowest kind) is one of the longest;
//   * 0.3 x the fraction of the next launch's clusters that cannot be resident
//     beside this launch's (those cannot start their set-up early).
int choose_splits(long long groups, long long T, int D) {
  const int n_sms = plan_sms();
  int best = 1;
  double best_cost = 1e300;
  for (int S = 1; S <= kAttnMaxSplits; ++S) {
    if (S > 1 && (groups * S > n_sms || groups > attn_max_clusters(S, D))) continue;
    const long long c = (T + S - 1) / S;
    double cost = static_cast<double>(c);
    if (S > 1) {
      const long long items = static_cast<long long>(attn_merge_rows(S)) * (D / 8);
      cost += 1.5 + 0.7 * static_cast<double>((items + 255) / 256 - 1);
      // the split of tile T - 1 under the ceil boundaries lo(s) = ceil(s T / S)
      long long lo_last = 0;
      for (int sp = S - 1; sp >= 0; --sp) {
        const long long lo = (sp * T + S - 1) / S;
        if (lo <= T - 1) {
          lo_last = lo;
          break;
        }
      }
      if (c >= 2 && T - lo_last == c) cost += 0.3;
      const long long blocked = 2 * groups - attn_max_clusters(S, D);
      if (blocked > 0) cost += 0.3 * static_cast<double>(blocked < groups ? blocked : groups) / groups;
    }
    if (cost <= best_cost) {
      best_cost = cost;
      best = S;
    }
  }
  return best;
}

bd_status plan_attention(const AttnDesc& d, AttnPlan* pl) {
  if (d.N < 1 || d.n_q < 1 || d.C < 0 || d.Hq < 1 || d.Hkv < 1 || d.priv_len < 0) return BD_ERR_INVALID_ARG;
  if (d.D != 64 && d.D != 128) return BD_ERR_UNSUPPORTED;
  if (d.Hq % d.Hkv != 0) return BD_ERR_UNSUPPORTED;
  if (d.q_pos != nullptr) {
    if (d.N != 1) return BD_ERR_INVALID_ARG;
  } else if (d.block_start == nullptr) {
    if (d.block_size < 1) return BD_ERR_INVALID_ARG;
  } else if (d.n_blocks < 1 || d.n_blocks > d.n_q) {
    return BD_ERR_INVALID_ARG;
  }
  if (d.num_splits < 0 || d.num_splits > kAttnMaxSplits) return BD_ERR_INVALID_ARG;
  if (d.rope.enabled && !(d.rope.theta > 0.f)) return BD_ERR_INVALID_ARG;
  if (d.kv_dtype != 0 && d.kv_dtype != BD_BF16 && d.kv_dtype != BD_E4M3) return BD_ERR_INVALID_ARG;
  if (d.kv_dtype == BD_E4M3 && (d.rope.enabled || d.q_pos != nullptr)) return BD_ERR_UNSUPPORTED;
  const long long G = d.Hq / d.Hkv;
  const long long per_roll = static_cast<long long>(d.n_q) * G;
  const long long rows = per_roll * d.N;
  if (rows > (1ll << 30)) return BD_ERR_UNSUPPORTED;
  pl->G = static_cast<int>(G);
  pl->rows_per_head = static_cast<int>(rows);
  pl->m_tiles = static_cast<int>((rows + kAttnBM - 1) / kAttnBM);
  pl->n_prefix_tiles = (d.C + kAttnBN - 1) / kAttnBN;
  // with the streaming mask the queries have no keys of their own
  const long long priv_tiles = d.q_pos ? 0 : (d.priv_len + d.n_q + kAttnBN - 1) / kAttnBN;
  const long long rolls_per_tile = (kAttnBM - 1) / per_roll + 2 < d.N ? (kAttnBM - 1) / per_roll + 2 : d.N;
  const long long max_tiles = pl->n_prefix_tiles + rolls_per_tile * priv_tiles;
  if (max_tiles > kAttnMaxTiles) return BD_ERR_UNSUPPORTED;
  pl->n_parts = 1;
  pl->part[0] = {0, pl->m_tiles, d.num_splits};
  if (d.num_splits == 0) {
    // spread the KV range of every (row tile, KV head) over the SMs as a cluster
    // of up to 16 CTAs, every cluster of the launch resident at once (one
    // wave), the split count chosen by choose_splits
    const long long groups = static_cast<long long>(pl->m_tiles) * d.Hkv;
    pl->part[0].splits = choose_splits(groups, max_tiles, d.D);
    const long long waves = groups / plan_sms();
    const int bulk = static_cast<int>(waves * plan_sms() / d.Hkv);  // whole waves of row tiles
    if (waves > 0 && bulk > 0 && bulk < pl->m_tiles) {
      const int tail_splits = choose_splits(static_cast<long long>(pl->m_tiles - bulk) * d.Hkv, max_tiles, d.D);
      if (tail_splits > 1) {
        pl->n_parts = 2;
        pl->part[0] = {0, bulk, 1};
        pl->part[1] = {bulk, pl->m_tiles - bulk, tail_splits};
      }
    }
  }
  int splits = 1;
  for (int i = 0; i < pl->n_parts; ++i) splits = pl->part[i].splits > splits ? pl->part[i].splits : splits;
  pl->splits = splits;
  // split partials: Hkv * m_tiles blocks of attn_part_bytes(splits, D); then,
  // with RoPE, the rotated prefix keys bf16 [Hkv, C, D]
  const size_t part_bytes = splits > 1 ? static_cast<size_t>(d.Hkv) * pl->m_tiles * attn_part_bytes(splits, d.D) : 0;
  pl->rope_off = (part_bytes + 255) / 256 * 256;
  const bool rope = d.rope.enabled && d.C > 0;
  pl->ws_bytes = rope ? pl->rope_off + static_cast<size_t>(d.Hkv) * d.C * d.D * 2 : part_bytes;
  return BD_OK;
}

// Parameters of the rotation of keys [0, C) of k (bf16 [Hkv, stride, D]) at
// k_pos - delta into out (bf16 [Hkv, C, D]): the frequencies theta^(-2d/D) in
// float64 and as 0.64 fixed-point turns, and 2 pi / 2^64 as float-float.
void rope_params(RopeParams* rp, const void* k, long long stride, void* out, int Hkv, int C, int D, const bd_rope& r) {
  std::memset(rp, 0, sizeof(*rp));
  rp->k = k;
  rp->out = out;
  rp->k_pos = r.k_pos;
  rp->Hkv = Hkv;
  rp->C = C;
  rp->D = D;
  rp->delta = r.delta;
  rp->stride = stride;
  const double two_pi = 6.283185307179586476925286766559;
  for (int i = 0; i < D / 2; ++i) {
    const double f = std::pow(static_cast<double>(r.theta), -2.0 * i / D);
    double x = f / two_pi;
    x -= std::floor(x);
    rp->turns[i] = static_cast<unsigned long long>(std::ldexp(x, 64));
    rp->freq[i] = f;
  }
  const double c = std::ldexp(two_pi, -64);
  rp->two_pi_64[0] = static_cast<float>(c);
  rp->two_pi_64[1] = static_cast<float>(c - static_cast<double>(rp->two_pi_64[0]));
}

bd_status run_attention(const AttnDesc& d, cudaStream_t stream) {
  AttnPlan pl;
  bd_status st = plan_attention(d, &pl);
  if (st != BD_OK) return st;
  if (!d.q || !d.pv || !d.pk || !d.rk || !d.rv || !d.o) return BD_ERR_INVALID_ARG;
  const bool kv8 = d.kv_dtype == BD_E4M3;
  if (kv8 && (!d.pk_exp || !d.pv_exp || !d.rk_exp || !d.rv_exp)) return BD_ERR_INVALID_ARG;
  if (!aligned(d.q, 16) || !aligned(d.o, 16) || !aligned(d.pk, 16) || !aligned(d.pv, 16) || !aligned(d.rk, 16) ||
      !aligned(d.rv, 16) || (d.lse && !aligned(d.lse, 4)))
    return BD_ERR_UNSUPPORTED;
  if (pl.ws_bytes > 0 && (d.ws == nullptr || d.ws_bytes < pl.ws_bytes || !aligned(d.ws, 256)))
    return BD_ERR_WORKSPACE;
  if ((st = check_device()) != BD_OK) return st;

  AttnParams p;
  std::memset(&p, 0, sizeof(p));
  p.q = d.q;
  p.o = d.o;
  p.lse = d.lse;
  p.part = pl.splits > 1 ? d.ws : nullptr;
  p.m_tiles = pl.m_tiles;
  p.m_tile0 = 0;
  p.block_start = d.block_start;
  p.dev_status = d.ds;
  p.N = d.N;
  p.n_q = d.n_q;
  p.Hq = d.Hq;
  p.Hkv = d.Hkv;
  p.G = pl.G;
  p.D = d.D;
  p.C = d.C;
  p.priv_len = d.priv_len;
  p.n_blocks = d.n_blocks;
  p.block_size = d.block_size;
  p.num_splits = pl.part[0].splits;
  p.rows_per_head = pl.rows_per_head;
  p.n_prefix_tiles = pl.n_prefix_tiles;
  // the rotated copy of a RoPE call is written by the kernel just before
  p.prefix_early = d.prefix_ready && !(d.rope.enabled && d.C > 0) ? 1 : 0;
  p.q_pos = d.q_pos;
  p.kpos = d.rope.k_pos;
  p.kdelta = d.rope.delta;
  p.wait_ns = wait_limit(d.wait_ns);
  if (kv8) {
    p.kv8 = 1;
    p.prefix_early = 0;
    p.pk_exp = d.pk_exp;
    p.pv_exp = d.pv_exp;
    p.rk_exp = d.rk_exp;
    p.rv_exp = d.rv_exp;
    p.p_exp_stride = d.p_exp_stride;
    p.r_exp_stride = d.r_exp_stride;
    p.r_exp_row0 = d.r_exp_row0;
  }
  const float scale = d.sm_scale > 0.f ? d.sm_scale : 1.0f / std::sqrt(static_cast<float>(d.D));
  p.scale_log2 = scale * 1.4426950408889634f;
  // RoPE: the pre-RoPE prefix keys are rotated once for the whole call into
  // the workspace, and the attention reads that copy
  const void* prefix_k = d.pk;
  long long prefix_k_stride = d.prefix_stride;
  RopeParams rp;
  const bool rope = d.rope.enabled && d.C > 0;
  if (rope) {
    rope_params(&rp, d.pk, d.prefix_stride, static_cast<char*>(d.ws) + pl.rope_off, d.Hkv, d.C, d.D, d.rope);
    prefix_k = rp.out;
    prefix_k_stride = d.C;
  }

  AttnMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  const uint64_t row_b = static_cast<uint64_t>(d.D) * 2;
  p.q_tma = (kAttnBM % pl.G) == 0 ? 1 : 0;
  if (p.q_tma) {
    // packed rows (position, g) of KV head h are G consecutive heads of each position
    const uint64_t dims[4] = {static_cast<uint64_t>(d.D), static_cast<uint64_t>(pl.G), static_cast<uint64_t>(d.Hkv),
                              static_cast<uint64_t>(d.N) * d.n_q};
    const uint64_t strides[3] = {row_b, row_b * pl.G, row_b * d.Hq};
    const uint32_t box[4] = {64, static_cast<uint32_t>(pl.G), 1, static_cast<uint32_t>(kAttnBM / pl.G)};
    if ((st = make_kv_map(&maps.q, d.q, 4, dims, strides, box)) != BD_OK) return st;
  }
  const uint64_t kv_row_b = kv8 ? static_cast<uint64_t>(d.D) : row_b;  // bytes of one K/V row
  if (d.C > 0) {
    const uint64_t dims[3] = {static_cast<uint64_t>(d.D), static_cast<uint64_t>(d.C), static_cast<uint64_t>(d.Hkv)};
    const uint64_t kstrides[2] = {kv_row_b, static_cast<uint64_t>(prefix_k_stride) * kv_row_b};
    const uint64_t strides[2] = {kv_row_b, static_cast<uint64_t>(d.prefix_stride) * kv_row_b};
    if ((st = make_kv_map(&maps.pk, prefix_k, 3, dims, kstrides, nullptr, kv8)) != BD_OK) return st;
    if ((st = make_kv_map(&maps.pv, d.pv, 3, dims, strides, nullptr, kv8)) != BD_OK) return st;
  }
  {
    const uint64_t dims[4] = {static_cast<uint64_t>(d.D), static_cast<uint64_t>(d.priv_len + d.n_q),
                              static_cast<uint64_t>(d.Hkv), static_cast<uint64_t>(d.N)};
    const uint64_t strides[3] = {kv_row_b, static_cast<uint64_t>(d.priv_stride) * kv_row_b,
                                 static_cast<uint64_t>(d.priv_stride) * kv_row_b * d.Hkv};
    if ((st = make_kv_map(&maps.rk, d.rk, 4, dims, strides, nullptr, kv8)) != BD_OK) return st;
    if ((st = make_kv_map(&maps.rv, d.rv, 4, dims, strides, nullptr, kv8)) != BD_OK) return st;
  }
  if (rope && launch_rope_prefix(rp, stream) != cudaSuccess) return BD_ERR_CUDA;
  for (int i = 0; i < pl.n_parts; ++i) {
    p.m_tile0 = pl.part[i].m_tile0;
    p.num_splits = pl.part[i].splits;
    if (launch_attention(p, maps, pl.part[i].m_tiles, stream) != cudaSuccess) return BD_ERR_CUDA;
  }
  return BD_OK;
}

AttnDesc desc_of(const bd_attn_args* a) {
  AttnDesc d;
  std::memset(&d, 0, sizeof(d));
  d.N = 1;
  d.q = a->q;
  d.pk = a->k;
  d.pv = a->v;
  d.prefix_stride = a->kv_stride;
  const size_t esz = a->kv_dtype == BD_E4M3 ? 1 : 2;  // bytes of a K/V element
  const size_t off = static_cast<size_t>(a->C > 0 ? a->C : 0) * (a->D > 0 ? a->D : 0) * esz;
  d.rk = a->k ? static_cast<const char*>(a->k) + off : nullptr;
  d.rv = a->v ? static_cast<const char*>(a->v) + off : nullptr;
  d.priv_stride = a->kv_stride;
  d.priv_len = 0;
  d.o = a->o;
  d.lse = a->lse;
  d.block_start = a->block_start;
  d.n_blocks = a->n_blocks;
  d.block_size = a->block_size;
  d.C = a->C;
  d.n_q = a->n_q;
  d.Hq = a->Hq;
  d.Hkv = a->Hkv;
  d.D = a->D;
  d.sm_scale = a->sm_scale;
  d.rope = a->rope;
  d.num_splits = a->num_splits;
  d.ws = a->workspace;
  d.ws_bytes = a->workspace_bytes;
  d.ds = a->dev_status;
  d.prefix_ready = a->prefix_ready;
  d.q_pos = a->q_pos;
  d.wait_ns = a->wait_limit_ns;
  d.kv_dtype = a->kv_dtype;
  d.pk_exp = d.rk_exp = a->k_exp;    // the active rows' exponents are those of rows C.. of the buffer
  d.pv_exp = d.rv_exp = a->v_exp;
  d.p_exp_stride = d.r_exp_stride = (a->kv_stride + kAttnBN - 1) / kAttnBN;
  d.r_exp_row0 = a->C;
  if (d.q_pos) {  // no active rows are read: point the private map at the cache itself
    d.rk = a->k;
    d.rv = a->v;
  }
  return d;
}

AttnDesc desc_of(const bd_fork_args* a) {
  AttnDesc d;
  std::memset(&d, 0, sizeof(d));
  d.N = a->N;
  d.q = a->q;
  d.pk = a->prefix_k;
  d.pv = a->prefix_v;
  d.prefix_stride = a->prefix_stride;
  d.rk = a->priv_k;
  d.rv = a->priv_v;
  d.priv_stride = a->priv_stride;
  d.priv_len = a->priv_len;
  d.o = a->o;
  d.lse = a->lse;
  d.block_start = a->block_start;
  d.n_blocks = a->n_blocks;
  d.block_size = a->block_size;
  d.C = a->C;
  d.n_q = a->n_q;
  d.Hq = a->Hq;
  d.Hkv = a->Hkv;
  d.D = a->D;
  d.sm_scale = a->sm_scale;
  d.rope = a->rope;
  d.num_splits = a->num_splits;
  d.ws = a->workspace;
  d.ws_bytes = a->workspace_bytes;
  d.ds = a->dev_status;
  d.prefix_ready = a->prefix_ready;
  d.wait_ns = a->wait_limit_ns;
  d.kv_dtype = a->kv_dtype;
  d.pk_exp = a->prefix_k_exp;
  d.pv_exp = a->prefix_v_exp;
  d.rk_exp = a->priv_k_exp;
  d.rv_exp = a->priv_v_exp;
  d.p_exp_stride = (a->prefix_stride + kAttnBN - 1) / kAttnBN;
  d.r_exp_stride = (a->priv_stride + kAttnBN - 1) / kAttnBN;
  d.r_exp_row0 = 0;
  return d;
}

// ------------------------------------------------------------------ unmask / verify

bd_status plan_unmask(const bd_unmask_args* a, int* chunks, int* elems, size_t* ws) {
  if (!a) return BD_ERR_INVALID_ARG;
  if (a->R < 1 || a->V < 1 || a->n_pos < 1 || a->n_blocks < 1 || a->n_blocks > a->n_pos) return BD_ERR_INVALID_ARG;
  if (a->n_pos > kMaxPos) return BD_ERR_UNSUPPORTED;
  if (a->logits_dtype != BD_F32 && a->logits_dtype != BD_BF16) return BD_ERR_INVALID_ARG;
  if (a->logits_ld < a->V || a->logits_ld % 8 != 0) return BD_ERR_INVALID_ARG;
  if (a->min_den < 1 || a->add_den < 1 || a->act_den < 1 || a->min_num < 0 || a->add_num < 0 || a->act_num < 0 ||
      a->k_fixed < 0)
    return BD_ERR_INVALID_ARG;
  if (a->R > kMaxVerifyRows) return BD_ERR_UNSUPPORTED;  // one CTA row per logits row (grid y)
  const int rows = a->R;
  vocab_split(rows, a->V, plan_sms(), chunks, elems);
  *ws = unmask_workspace_bytes(a->R);
  return BD_OK;
}

bd_status plan_verify(const bd_verify_args* a, int* chunks, int* elems, size_t* ws) {
  if (!a) return BD_ERR_INVALID_ARG;
  if (a->n_seq < 1 || a->L < 1 || a->n_rows < 1 || a->n_rows > a->L + 1 || a->V < 1) return BD_ERR_INVALID_ARG;
  if (a->L > 1024) return BD_ERR_UNSUPPORTED;
  if (static_cast<long long>(a->n_seq) * a->n_rows > kMaxVerifyRows || a->n_seq > kMaxVerifySeqs)
    return BD_ERR_UNSUPPORTED;
  if (a->logits_dtype != BD_F32 && a->logits_dtype != BD_BF16) return BD_ERR_INVALID_ARG;
  if (a->logits_ld < a->V || a->logits_ld % 8 != 0) return BD_ERR_INVALID_ARG;
  if (a->noise && !(a->temperature > 0.f)) return BD_ERR_INVALID_ARG;
  vocab_split(a->n_seq * a->n_rows, a->V, plan_sms(), chunks, elems);
  *ws = verify_workspace_bytes(a->n_seq, a->n_rows);
  return BD_OK;
}

}  // namespace

extern "C" {

size_t bd_attn_workspace_size(const bd_attn_args* a) {
  if (!a) return 0;
  AttnPlan pl;
  return plan_attention(desc_of(a), &pl) == BD_OK ? pl.ws_bytes : 0;
}

size_t bd_fork_workspace_size(const bd_fork_args* a) {
  if (!a) return 0;
  AttnPlan pl;
  return plan_attention(desc_of(a), &pl) == BD_OK ? pl.ws_bytes : 0;
}

bd_status bd_block_causal_attn(const bd_attn_args* a, void* stream) {
  if (!a || !a->q || !a->k || !a->v || !a->o) return BD_ERR_INVALID_ARG;
  if (a->kv_stride < static_cast<long long>(a->C) + (a->q_pos ? 0 : a->n_q)) return BD_ERR_INVALID_ARG;
  if (a->q_pos && (!aligned(a->q_pos, 4) || (a->rope.k_pos && !aligned(a->rope.k_pos, 16)))) return BD_ERR_UNSUPPORTED;
  return run_attention(desc_of(a), static_cast<cudaStream_t>(stream));
}

bd_status bd_fork_rollouts(const bd_fork_args* a, void* stream) {
  if (!a || !a->q || !a->prefix_k || !a->prefix_v || !a->priv_k || !a->priv_v || !a->o) return BD_ERR_INVALID_ARG;
  if (a->C > 0 && a->prefix_stride < a->C) return BD_ERR_INVALID_ARG;
  if (a->priv_stride < static_cast<long long>(a->priv_len) + a->n_q) return BD_ERR_INVALID_ARG;
  return run_attention(desc_of(a), static_cast<cudaStream_t>(stream));
}

bd_status bd_stream_insert(const bd_stream_insert_args* a, void* stream) {
  if (!a || !a->k_cache || !a->v_cache || !a->k_pos || !a->new_k || !a->new_v || !a->new_pos)
    return BD_ERR_INVALID_ARG;
  if (a->views < 1 || a->frames < 1 || a->per_frame < 1 || a->Hkv < 1 || a->slot < 0 || a->slot >= a->frames)
    return BD_ERR_INVALID_ARG;
  if (a->D != 64 && a->D != 128) return BD_ERR_UNSUPPORTED;
  const long long window = static_cast<long long>(a->views) * a->frames * a->per_frame;
  if (window > (1ll << 30) || a->cache_stride < window) return BD_ERR_INVALID_ARG;
  if (!aligned(a->k_cache, 16) || !aligned(a->v_cache, 16) || !aligned(a->new_k, 16) || !aligned(a->new_v, 16) ||
      !aligned(a->k_pos, 4) || !aligned(a->new_pos, 4))
    return BD_ERR_UNSUPPORTED;
  bd_status st = check_device();
  if (st != BD_OK) return st;
  StreamInsertParams p;
  p.k_cache = a->k_cache;
  p.v_cache = a->v_cache;
  p.k_pos = a->k_pos;
  p.new_k = a->new_k;
  p.new_v = a->new_v;
  p.new_pos = a->new_pos;
  p.views = a->views;
  p.frames = a->frames;
  p.per_frame = a->per_frame;
  p.slot = a->slot;
  p.Hkv = a->Hkv;
  p.D = a->D;
  p.stride = a->cache_stride;
  return launch_stream_insert(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? BD_OK : BD_ERR_CUDA;
}

bd_status bd_rope_keys(const bd_rope_keys_args* a, void* stream) {
  if (!a || !a->k || !a->out) return BD_ERR_INVALID_ARG;
  if (a->Hkv < 1 || a->C < 0 || a->k_stride < a->C || !(a->rope.theta > 0.f)) return BD_ERR_INVALID_ARG;
  if (a->D != 64 && a->D != 128) return BD_ERR_UNSUPPORTED;
  if (!aligned(a->k, 16) || !aligned(a->out, 16) || (a->rope.k_pos && !aligned(a->rope.k_pos, 4)))
    return BD_ERR_UNSUPPORTED;
  const char* k0 = static_cast<const char*>(a->k);
  const char* k1 = k0 + static_cast<size_t>(a->Hkv) * a->k_stride * a->D * 2;
  const char* o0 = static_cast<const char*>(a->out);
  const char* o1 = o0 + static_cast<size_t>(a->Hkv) * a->C * a->D * 2;
  if (o0 < k1 && k0 < o1) return BD_ERR_INVALID_ARG;  // out overlaps k
  bd_status st = check_device();
  if (st != BD_OK) return st;
  if (a->C == 0) return BD_OK;
  RopeParams rp;
  rope_params(&rp, a->k, a->k_stride, a->out, a->Hkv, a->C, a->D, a->rope);
  return launch_rope_prefix(rp, static_cast<cudaStream_t>(stream)) == cudaSuccess ? BD_OK : BD_ERR_CUDA;
}

size_t bd_unmask_workspace_size(const bd_unmask_args* a) {
  int c, e;
  size_t ws = 0;
  return plan_unmask(a, &c, &e, &ws) == BD_OK ? ws : 0;
}

}  // extern "C"

namespace {

// Every host-side check of an unmask call (shapes, pointers, alignment,
// workspace, device), then its kernel parameters; nothing is enqueued.
bd_status prepare_unmask(const bd_unmask_args* a, UnmaskParams* out) {
  int chunks, elems;
  size_t ws;
  bd_status st = plan_unmask(a, &chunks, &elems, &ws);
  if (st != BD_OK) return st;
  if (!a->logits || !a->logit_row || !a->block_start || !a->state || !a->tokens || !a->commit || !a->n_committed ||
      !a->status)
    return BD_ERR_INVALID_ARG;
  if (!aligned(a->logits, 16)) return BD_ERR_UNSUPPORTED;
  if (!a->workspace || a->workspace_bytes < ws || !aligned(a->workspace, 256)) return BD_ERR_WORKSPACE;
  if ((st = check_device()) != BD_OK) return st;
  UnmaskParams& p = *out;
  std::memset(&p, 0, sizeof(p));
  p.logits = a->logits;
  p.dtype = a->logits_dtype;
  p.ld = a->logits_ld;
  p.R = a->R;
  p.V = a->V;
  p.logit_row = a->logit_row;
  p.n_pos = a->n_pos;
  p.block_start = a->block_start;
  p.n_blocks = a->n_blocks;
  p.state = a->state;
  p.tokens = a->tokens;
  p.tau_full = a->tau_full;
  p.tau_half = a->tau_half;
  p.min_num = a->min_num;
  p.min_den = a->min_den;
  p.k_fixed = a->k_fixed;
  p.add_num = a->add_num;
  p.add_den = a->add_den;
  p.act_num = a->act_num;
  p.act_den = a->act_den;
  p.commit = a->commit;
  p.n_committed = a->n_committed;
  p.status = a->status;
  p.pred = a->pred;
  p.conf = a->conf;
  p.lse = a->lse;
  p.write_draft = a->write_draft;
  p.dev_status = a->dev_status;
  p.wait_ns = wait_limit(a->wait_limit_ns);
  char* w = static_cast<char*>(a->workspace);
  p.grid_ticket = reinterpret_cast<unsigned*>(w);
  p.row_res = reinterpret_cast<float4*>(w + unmask_counter_bytes());
  p.chunks = chunks;
  p.chunk_elems = elems;
  return BD_OK;
}

}  // namespace

extern "C" {

bd_status bd_unmask_step(const bd_unmask_args* a, void* stream) {
  UnmaskParams p;
  const bd_status st = prepare_unmask(a, &p);
  if (st != BD_OK) return st;
  return launch_unmask(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? BD_OK : BD_ERR_CUDA;
}

size_t bd_verify_workspace_size(const bd_verify_args* a) {
  int c, e;
  size_t ws = 0;
  return plan_verify(a, &c, &e, &ws) == BD_OK ? ws : 0;
}

bd_status bd_spec_verify(const bd_verify_args* a, void* stream) {
  int chunks, elems;
  size_t ws;
  bd_status st = plan_verify(a, &chunks, &elems, &ws);
  if (st != BD_OK) return st;
  if (!a->tokens || !a->state || !a->ar_logits || !a->accepted_len || !a->bonus || !a->bonus_pos)
    return BD_ERR_INVALID_ARG;
  if (!aligned(a->ar_logits, 16) || (a->noise && !aligned(a->noise, 16))) return BD_ERR_UNSUPPORTED;
  if (!a->workspace || a->workspace_bytes < ws || !aligned(a->workspace, 256)) return BD_ERR_WORKSPACE;
  if ((st = check_device()) != BD_OK) return st;
  VerifyParams p;
  std::memset(&p, 0, sizeof(p));
  p.n_seq = a->n_seq;
  p.L = a->L;
  p.tokens = a->tokens;
  p.state = a->state;
  p.logits = a->ar_logits;
  p.dtype = a->logits_dtype;
  p.ld = a->logits_ld;
  p.n_rows = a->n_rows;
  p.V = a->V;
  p.noise = a->noise;
  p.inv_temp = a->noise ? 1.0f / a->temperature : 1.0f;
  p.accepted_len = a->accepted_len;
  p.bonus = a->bonus;
  p.bonus_pos = a->bonus_pos;
  p.dev_status = a->dev_status;
  p.wait_ns = wait_limit(a->wait_limit_ns);
  char* w = static_cast<char*>(a->workspace);
  p.seq_ticket = reinterpret_cast<unsigned*>(w);
  p.row_res = reinterpret_cast<float4*>(w + verify_counter_bytes());
  p.chunks = chunks;
  p.chunk_elems = elems;
  return launch_verify(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? BD_OK : BD_ERR_CUDA;
}

const char* bd_status_string(bd_status s) {
  switch (s) {
    case BD_OK: return "ok";
    case BD_ERR_INVALID_ARG: return "invalid argument";
    case BD_ERR_UNSUPPORTED: return "unsupported shape, alignment or device";
    case BD_ERR_WORKSPACE: return "workspace missing or too small";
    case BD_ERR_CUDA: return "CUDA call failed";
    case BD_ERR_TIMEOUT: return "a device-side bounded wait expired";
    case BD_ERR_DEVICE_INPUT: return "the device found an inconsistent input";
  }
  return "unknown status";
}

bd_status bd_check(const int32_t* dev_status, void* stream) {
  if (!dev_status) return BD_ERR_INVALID_ARG;
  int32_t h = 0;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return BD_ERR_CUDA;
  if (cudaMemcpy(&h, dev_status, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return BD_ERR_CUDA;
  if (h & BD_DEV_TIMEOUT) return BD_ERR_TIMEOUT;
  if (h & BD_DEV_BAD_INPUT) return BD_ERR_DEVICE_INPUT;
  return BD_OK;
}

const char* bd_version(void) { return "0.1.0"; }

}  // extern "C"

// ------------------------------------------------------------------ allocation-free unmask step
//
// For callers that cannot allocate device memory, the scratch of one unmask
// step lives in this fixed array, which every GPU that loads the library holds
// until the process exits.  Host code must not pass the array's name to a
// kernel (on the host it is only a stand-in for the symbol): its device address
// is looked up once per device with cudaGetSymbolAddress and cached.

namespace {

static __device__ __align__(256) unsigned char g_unmask_scratch[BD_UNMASK_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
void* g_scratch_addr[64];  // device address of g_unmask_scratch on each device, once looked up

}  // namespace

extern "C" bd_status bd_unmask_step_noalloc(const bd_unmask_args* a, void* stream) {
  int chunks, elems;
  size_t need;
  bd_status st = plan_unmask(a, &chunks, &elems, &need);
  if (st != BD_OK) return st;
  if (need > BD_UNMASK_NOALLOC_SCRATCH_BYTES) return BD_ERR_WORKSPACE;
  if ((st = check_device()) != BD_OK) return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BD_ERR_CUDA;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_unmask_scratch) != cudaSuccess || ptr == nullptr) return BD_ERR_CUDA;
      g_scratch_addr[dev] = ptr;
    }
    scratch = g_scratch_addr[dev];
  }
  bd_unmask_args b = *a;
  b.workspace = scratch;
  b.workspace_bytes = BD_UNMASK_NOALLOC_SCRATCH_BYTES;
  // every argument is checked before anything is enqueued
  UnmaskParams p;
  if ((st = prepare_unmask(&b, &p)) != BD_OK) return st;
  // The counter words must start at zero; a call cut short may have left them set.
  if (cudaMemsetAsync(scratch, 0, unmask_counter_bytes(), static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return BD_ERR_CUDA;
  return launch_unmask(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? BD_OK : BD_ERR_CUDA;
}
