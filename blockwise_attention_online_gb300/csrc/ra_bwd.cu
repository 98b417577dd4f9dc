// Backward pass of the ring forward on the 5th-generation tensor cores:
// dQ, and dK, dV of every key/value chunk, in fp32.
//
// "Ring Attention: Distributed Reads with Online Softmax", section "Backward
// must aggregate shared dependencies": a query row's gradient reaches every
// key/value shard it attended to and has to be summed per shard for the
// shard's owner; the probability tiles may be recomputed, with the forward's
// scale and masks. Here the forward's row statistics (m, l) fix every
// probability, P = exp(s - m) / l = exp2(s * scale * log2(e) - lse2), so each
// tile is recomputed independently of the visit order:
//
//   dV_c = P_c^T dO              dP_c = dO V_c^T
//   dS_c = P_c * (dP_c - delta)  delta = rowsum(dO * O)
//   dK_c = scale dS_c^T Q        dQ   = scale sum_c dS_c K_c
//
// Three launches on the caller's stream:
//   bwd_prep_kernel    per query row lse2 and delta, per query tile the
//                      column data of the dK/dV CTAs and its key-window bounds
//   bwd_kernel<D>      two kinds of CTA in one grid:
//     bwd_dkv_tile     one per (batch, key/value head, 128-row key tile):
//                      walks every live query tile of the heads that read it
//                      and accumulates dK, dV in TMEM (the per-shard sum)
//     bwd_dq_tile      one per (batch, query head, 128-row query tile):
//                      walks every live key tile and accumulates dQ in TMEM
//
// Warp roles of both kinds of CTA (384 threads): warp 0 TMA producer,
// warp 1 MMA warp (waits warp-uniformly, one elected lane issues), warps 2-3
// idle, warps 4-11 the elementwise work: one TMEM lane (= tile row) per
// thread, warpgroup h on columns [64h, 64h + 64) of every 128-column tile (no
// step of the backward reduces across columns, so the halves never meet).
// Every mbarrier wait is bounded (see ra_wait.cuh).
#include <cuda_runtime.h>
#include <stdint.h>

#include "ra.h"
#include "ra_plan.h"
#include "ra_ptx.cuh"
#include "ra_wait.cuh"

namespace ra {
namespace {

using namespace ptx;

constexpr int kBwdThreads = 384;
constexpr float kInf = __builtin_huge_valf();
constexpr float kLog2e = 1.4426950408889634f;

enum : int {
  kSiteBwdKv = 31, kSiteBwdStage = 32, kSiteBwdEmpty = 33, kSiteBwdSdp = 34, kSiteBwdDs = 35,
  kSiteBwdAcc = 36
};

// kDocs: the dK/dV CTAs of a launch with packed documents walk only the
// query tiles whose rows' key windows meet their key tile.
template <int D, bool kDocs = true>
struct BwdCfg {
  static constexpr int kBoxBytes = 128 * 128;     // 128 rows x 64 bf16 (one swizzle atom wide)
  static constexpr int kBoxes = (D + 63) / 64;    // D = 96: the second box is half zero fill
  static constexpr int kTileBytes = kBoxes * kBoxBytes;  // one 128-row bf16 tile
  // shared memory of a dK/dV CTA: K and V resident; two stages, each of a Q
  // and a dO tile and the query tile's column data (kColAuxBytes: the two
  // column-bias tiles, then the key windows); the constant tile of ones the
  // biases are multiplied with; barriers
  static constexpr int kRes0 = 0, kRes1 = kTileBytes;
  static constexpr int kStage0 = 2 * kTileBytes;
  static constexpr int kStageBytes = 2 * kTileBytes;
  // A bias tile is a K = 16 operand of 128 rows (4 KB, no swizzle): row n
  // holds a value of query column n as the sum of three bf16 numbers in K
  // slots 0-2, the other slots zero. Stage s: [-lse2 / c, -delta, windows].
  static constexpr int kBiasBytes = 128 * 16 * 2;
  static constexpr int kAux0 = kStage0 + 2 * kStageBytes;
  static constexpr int kAuxBytes = kColAuxBytes;
  static constexpr int kOnes = kAux0 + 2 * kAuxBytes;     // rows (1, 1, 1, 0, ...)
  static constexpr int kBar = kOnes + kBiasBytes;
  static constexpr int kBarBytes = 256;
  static constexpr int kSmemBytes = kBar + kBarBytes + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  static_assert(kAux0 % 1024 == 0 && kAuxBytes % 1024 == 0, "bias tiles stay aligned");
  // epilogue: dK and dV as padded row-major fp32 tiles over the K/V and stage
  // buffers (free once every product is complete)
  static constexpr int kEpiPitch = D + 4;  // floats per staged row
  static constexpr int kEpiK = 0, kEpiV = 128 * kEpiPitch * 4;
  static_assert(kEpiV + 128 * kEpiPitch * 4 <= kAux0, "epilogue tiles fit the free buffers");
};

// Stores rows [0, nrows) of a staged fp32 tile (row pitch D + 4 floats) to
// consecutive rows of `dst` (D floats each): the 256 elementwise threads,
// warp e taking rows e, e + 8, ..., each lane 16 bytes of the row, so every
// store instruction writes whole rows.
template <int D>
__device__ __forceinline__ void store_staged_rows(const float* stage, float* dst, int nrows, int e,
                                                  int lane) {
  if (lane >= D / 4) return;
  for (int rr = e; rr < nrows; rr += 8)
    reinterpret_cast<float4*>(dst + int64_t(rr) * D)[lane] =
        reinterpret_cast<const float4*>(stage + rr * (D + 4))[lane];
}


// Non-blocking check of an mbarrier phase, the same answer for the whole warp
// (lane 0 tests, the warp follows).
__device__ __forceinline__ bool warp_phase_done(uint32_t bar, uint32_t parity) {
  uint32_t done = 0;
  if ((threadIdx.x & 31) == 0) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
  }
  return __shfl_sync(0xffffffffu, done, 0) != 0;
}

// Chunk tables: the plan's own arrays, or their device-resident copies (read
// in separate branches, see ld_kvseg).
__device__ __forceinline__ KvSeg bspan(const BwdPlan& p, int k) {
  if (p.ext_ks != nullptr) return ld_kvseg(p.ext_ks + k);
  return p.ks[k];
}
__device__ __forceinline__ int btile_begin(const BwdPlan& p, int k) {
  if (p.ext_ktb != nullptr) return __ldg(p.ext_ktb + k);
  return p.kseg_tile_begin[k];
}
__device__ __forceinline__ QPiece bqpiece(const BwdPlan& p, int i) {
  if (p.ext_qp != nullptr) return ld_qpiece(p.ext_qp + i);
  return p.qp[i];
}
__device__ __forceinline__ const CUtensorMap* bkmap(const BwdPlan& p, int c) {
  return p.ext_kmap ? p.ext_kmap + c : &p.kmap[c];
}
__device__ __forceinline__ const CUtensorMap* bvmap(const BwdPlan& p, int c) {
  return p.ext_vmap ? p.ext_vmap + c : &p.vmap[c];
}
// Before the first TMA copy through a chunk's maps: device-resident maps
// were written by a copy from the host (generic proxy).
__device__ __forceinline__ void bwd_fence_maps(const BwdPlan& p, int c) {
  if (p.ext_kmap != nullptr) {
    fence_tmap_acquire(p.ext_kmap + c);
    fence_tmap_acquire(p.ext_vmap + c);
  }
}

// Byte offset of row n's K slots 0-7 in a no-swizzle K = 16 operand tile
// (8-row groups of two 128-byte core matrices; slots 8-15 at +128 stay zero).
__device__ __forceinline__ uint32_t bias_row_offset(int n) { return (n >> 3) * 256 + (n & 7) * 16; }

// x as hi + mid + lo, three bf16 numbers (error below 2^-26 |x|), in K slots
// 0-2 of a row; the products with a row of ones add them up in fp32.
__device__ __forceinline__ uint4 bias_split3(float x) {
  const uint32_t h = pack_bf16x2(x, 0.f) & 0xffffu;
  const float r1 = x - __uint_as_float(h << 16);
  const uint32_t m = pack_bf16x2(r1, 0.f) & 0xffffu;
  const float r2 = r1 - __uint_as_float(m << 16);
  const uint32_t l = pack_bf16x2(r2, 0.f) & 0xffffu;
  return make_uint4(h | (m << 16), l, 0u, 0u);
}

__device__ __forceinline__ int bwd_row_position(const BwdPlan& p, int row) {
  int lo = 0, hi = p.n_qpieces - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (bqpiece(p, mid).row0 <= row) lo = mid; else hi = mid - 1;
  }
  const QPiece q = bqpiece(p, lo);
  return q.pos0 + q.step * (row - q.row0);
}

// Key tiles [tb, te) of span k holding a position inside the key window
// [lo, hi] of some row of a query tile.
__device__ __forceinline__ void bwd_live_tiles(const BwdPlan& p, int k, int lo, int hi, int& tb,
                                               int& te) {
  const KvSeg s = bspan(p, k);
  if (!p.causal && p.n_docs == 0) {
    tb = 0;
    te = s.ntiles;
    return;
  }
  live_range(s.pos0, s.step, s.len, lo, hi, tb, te);
}

// ------------------------------------------------------------ preparation
// One block of 128 threads per (batch x query head, 128-row query tile), one
// thread per query row (the rows past Sq of the last tile included):
//   delta = sum_d dO * O (O as the forward wrote it) and
//   lse2 = m log2(e) + log2(l) (+inf for a row that sees no key);
//   the dK/dV CTAs' column data of the tile, laid out as it will lie in
//   shared memory (kColAuxBytes per tile): the bias rows -lse2 / c and
//   -delta, each as three bf16 parts (-1e30 for a row that sees no key or
//   lies past Sq, so that its probabilities are 0), and the row's key window;
//   for batch x head 0, the bounds of the tile's key windows (x: lowest lo,
//   y: highest hi, z: highest lo, w: lowest hi): a key tile inside [z, w] is
//   visible to every row, one outside [x, y] to none.
template <int D>
__global__ void __launch_bounds__(128) bwd_prep_kernel(const __grid_constant__ BwdPlan p,
                                                       const void* o, int o_fp32, int64_t o_sb,
                                                       int64_t o_sh, int64_t o_sr,
                                                       const uint16_t* dout, const float* m,
                                                       const float* l, float* lse2, float* delta,
                                                       int4* qtile_pos, uint8_t* colaux) {
  const int qt = blockIdx.x % p.n_qtiles;
  const int bh = blockIdx.x / p.n_qtiles;
  const int b = bh / p.Hq, h = bh - b * p.Hq;
  const int n = threadIdx.x;
  const int row = 128 * qt + n;
  const bool valid = row < p.Sq;
  // delta of the tile's rows: eight lanes per row (each load instruction of a
  // warp covers four consecutive rows), partial sums added by shuffles
  __shared__ float sdl[128];
  {
    const int warp = n >> 5, lane = n & 31, grp = lane >> 3, l8 = lane & 7;
    constexpr int kU2 = D / 32;  // 4-element pieces per lane
#pragma unroll 1
    for (int it = 0; it < 8; ++it) {
      const int rl = warp * 32 + 4 * it + grp;
      const int rr = 128 * qt + rl;
      float acc = 0.f;
      if (rr < p.Sq) {
        const int64_t off = int64_t(b) * o_sb + int64_t(h) * o_sh + int64_t(rr) * o_sr;
        const uint2* g2 = reinterpret_cast<const uint2*>(dout + off) + l8 * kU2;
#pragma unroll
        for (int e = 0; e < kU2; ++e) {
          const uint2 gv = g2[e];
          const float g0 = __uint_as_float(gv.x << 16), g1 = __uint_as_float(gv.x & 0xffff0000u);
          const float g2v = __uint_as_float(gv.y << 16), g3 = __uint_as_float(gv.y & 0xffff0000u);
          if (o_fp32) {
            const float4 ov = reinterpret_cast<const float4*>(static_cast<const float*>(o) + off)[l8 * kU2 + e];
            acc = fmaf(g0, ov.x, fmaf(g1, ov.y, fmaf(g2v, ov.z, fmaf(g3, ov.w, acc))));
          } else {
            const uint2 ov = reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(o) + off)[l8 * kU2 + e];
            acc = fmaf(g0, __uint_as_float(ov.x << 16),
                       fmaf(g1, __uint_as_float(ov.x & 0xffff0000u),
                            fmaf(g2v, __uint_as_float(ov.y << 16),
                                 fmaf(g3, __uint_as_float(ov.y & 0xffff0000u), acc))));
          }
        }
      }
      acc += __shfl_xor_sync(0xffffffffu, acc, 4);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      if (l8 == 0) sdl[rl] = acc;
    }
  }
  __syncthreads();
  float dl = 0.f, l2 = kInf;
  int lo = 0x7fffffff, hi = int(0x80000000);  // an empty window
  if (valid) {
    dl = sdl[n];
    const int64_t srow = int64_t(bh) * p.Sq + row;
    const float lr = l[srow];
    l2 = lr > 0.f ? fmaf(m[srow], kLog2e, log2f(lr)) : kInf;
    delta[srow] = dl;
    lse2[srow] = l2;
    if (p.causal || p.n_docs > 0) {
      key_window(p, bwd_row_position(p, row), lo, hi);
    } else {
      lo = 0;
      hi = 0x7fffffff;
    }
  }
  uint8_t* tile = colaux + (int64_t(bh) * p.n_qtiles + qt) * int64_t(kColAuxBytes);
  const uint32_t boff = bias_row_offset(n);
  *reinterpret_cast<uint4*>(tile + boff) = bias_split3(l2 < kInf ? -l2 / p.scale_log2 : -1e30f);
  *reinterpret_cast<uint4*>(tile + boff + 128) = make_uint4(0u, 0u, 0u, 0u);
  *reinterpret_cast<uint4*>(tile + 4096 + boff) = bias_split3(-dl);
  *reinterpret_cast<uint4*>(tile + 4096 + boff + 128) = make_uint4(0u, 0u, 0u, 0u);
  reinterpret_cast<int2*>(tile + 8192)[n] = make_int2(lo, hi);
  if (bh == 0) {
    // the same positions for every batch element and head: one block per tile
    __shared__ int4 red[4];
    int4 w = valid ? make_int4(lo, hi, lo, hi) : make_int4(0x7fffffff, -1, -1, 0x7fffffff);
    w.x = __reduce_min_sync(0xffffffffu, w.x);
    w.y = __reduce_max_sync(0xffffffffu, w.y);
    w.z = __reduce_max_sync(0xffffffffu, w.z);
    w.w = __reduce_min_sync(0xffffffffu, w.w);
    if ((n & 31) == 0) red[n >> 5] = w;
    __syncthreads();
    if (n == 0) {
      for (int i = 1; i < 4; ++i) {
        w.x = min(w.x, red[i].x);
        w.y = max(w.y, red[i].y);
        w.z = max(w.z, red[i].z);
        w.w = min(w.w, red[i].w);
      }
      qtile_pos[qt] = w;
    }
  }
}

// ------------------------------------------------------------ shared pieces
struct BwdBars {
  uint32_t res_full, st_full0, st_empty0, sdp_full, ew_done, acc_full, done, s_free;  // stage s: + 8 s
  uint32_t* tmem_slot;
  volatile int* abort_flag;
};

template <int D, bool kDocs = true, bool kBias = false>
__device__ __forceinline__ void bwd_setup(uint8_t* smem_raw, uint32_t& base, uint8_t*& gbase,
                                          BwdBars& bb) {
  using C = BwdCfg<D, kDocs>;
  const uint32_t raw = smem_addr(smem_raw);
  base = (raw + 1023u) & ~1023u;
  gbase = smem_raw + (base - raw);
  if constexpr (kBias) {
    // the ones tile: 1.0 in K slots 0-2 of every row, the other slots zero
    for (int n = threadIdx.x; n < 128; n += blockDim.x) {
      *reinterpret_cast<uint4*>(gbase + C::kOnes + bias_row_offset(n)) =
          make_uint4(0x3f803f80u, 0x00003f80u, 0u, 0u);
      *reinterpret_cast<uint4*>(gbase + C::kOnes + bias_row_offset(n) + 128) = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
  }
  const uint32_t bars = base + C::kBar;
  bb.res_full = bars;
  bb.st_full0 = bars + 8;
  bb.st_empty0 = bars + 24;
  bb.sdp_full = bars + 40;
  bb.ew_done = bars + 48;
  bb.acc_full = bars + 56;
  bb.done = bars + 64;
  bb.s_free = bars + 72;
  bb.tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kBar + 80);
  bb.abort_flag = reinterpret_cast<volatile int*>(gbase + C::kBar + 84);
  if (threadIdx.x == 0) {
    mbar_init(bb.res_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bb.st_full0 + 8 * s, 1);  // the copies' transaction count
      mbar_init(bb.st_empty0 + 8 * s, 1);
    }
    mbar_init(bb.sdp_full, 1);
    mbar_init(bb.ew_done, 256);
    mbar_init(bb.acc_full, 1);
    mbar_init(bb.done, 1);
    mbar_init(bb.s_free, 256);
    *bb.abort_flag = 0;
    fence_mbar_init();
  }
  if ((threadIdx.x >> 5) == 1) {
    tmem_alloc(smem_addr(bb.tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}

__device__ __forceinline__ void bwd_teardown(uint32_t tmem) {
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if ((threadIdx.x >> 5) == 1) tmem_dealloc(tmem, 512);
}

// Issue one 128 x 128 x D product D[tmem] = A B^T, both operands K-major in
// shared memory (the layout TMA writes for a [rows, D] tile).
// acc: add to what the accumulator holds (a bias) instead of overwriting it.
template <int D>
__device__ __forceinline__ void issue_abt(uint32_t d_tmem, uint32_t sa, uint32_t sb,
                                          bool acc = false) {
  using C = BwdCfg<D>;
  constexpr uint32_t kId = idesc_bf16_f32(128, 128, 0, 0);
  const uint64_t ad = sdesc_sw128(sa, 16, 1024), bd = sdesc_sw128(sb, 16, 1024);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t off = uint64_t(((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4);
    mma_ss(d_tmem, ad + off, bd + off, kId, (acc || kk > 0) ? 1u : 0u);
  }
}

// D[tmem] = ones . bias^T: every row of the 128 x 128 accumulator receives the
// per-column bias (K = 16, both operands without swizzle).
__device__ __forceinline__ void issue_bias(uint32_t d_tmem, uint32_t s_ones, uint32_t s_bias) {
  constexpr uint32_t kId = idesc_bf16_f32(128, 128, 0, 0);
  mma_ss(d_tmem, sdesc_noswizzle(s_ones, 128, 256), sdesc_noswizzle(s_bias, 128, 256), kId, 0u);
}

// D[tmem] (+)= A[tmem] B with A 128 x 128 bf16 in TMEM and B a [128 rows (the
// contraction), D] tile in shared memory (MN-major). Contraction index
// 64h + x of A sits in column a_tmem + 64h + x/2: each elementwise warpgroup
// h writes its half inside the columns it read.
template <int D>
__device__ __forceinline__ void issue_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint32_t sb,
                                             bool acc) {
  using C = BwdCfg<D>;
  constexpr uint32_t kId = idesc_bf16_f32(128, D, 0, 1);
  const uint64_t bd = sdesc_sw128(sb, C::kBoxBytes, 1024);
#pragma unroll
  for (int kk = 0; kk < 128 / 16; ++kk)
    mma_ts(d_tmem, a_tmem + 64 * (kk >> 2) + 8 * (kk & 3), bd + uint64_t((kk * 16 * 128) >> 4), kId,
           (acc || kk > 0) ? 1u : 0u);
}

// ------------------------------------------------------------ dK, dV
// The query tiles a key tile sees: heads hkv*g .. hkv*g + g - 1, every tile
// whose rows' key windows meet the key tile's positions [kmin, kmax] (all
// when neither causal nor packed).
template <bool kDocs>
struct QWalk {
  int idx, n, nqt, h0;
  __device__ __forceinline__ bool next(const BwdPlan& p, int kmin, int kmax, int& h, int& qt) {
    while (idx < n) {
      const int i = idx++;
      qt = i % nqt;
      h = h0 + i / nqt;
      if constexpr (kDocs) {
        const int4 w = p.qtile_pos[qt];
        if (w.y >= kmin && w.x <= kmax) return true;
      } else {
        if (!p.causal || p.qtile_pos[qt].y >= kmin) return true;
      }
    }
    return false;
  }
};

template <int D, bool kDocs>
__device__ __forceinline__ void bwd_dkv_tile(const BwdPlan& p, int cta) {
  using C = BwdCfg<D, kDocs>;
  extern __shared__ uint8_t smem_raw[];
  uint32_t base;
  uint8_t* gbase;
  BwdBars bb;
  bwd_setup<D, kDocs, true>(smem_raw, base, gbase, bb);
  const uint32_t tmem = *bb.tmem_slot;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned long long budget = p.timeout_ns;

  // this CTA's key tile
  int u = cta;
  const int gt = u % p.n_ktiles;
  u /= p.n_ktiles;
  const int hkv = u % p.Hkv, b = u / p.Hkv;
  int ks = 0;  // last span whose first tile is at or before gt
  {
    int hi = p.n_kvsegs - 1;
    while (ks < hi) {
      const int mid = (ks + hi + 1) >> 1;
      if (btile_begin(p, mid) <= gt) ks = mid; else hi = mid - 1;
    }
  }
  const KvSeg sg = bspan(p, ks);
  const int kt = gt - btile_begin(p, ks);
  const int krow0 = sg.row0 + 128 * kt;                 // first row within the chunk
  const int kvalid = min(128, sg.len - 128 * kt);       // rows of the tile that exist
  const int kmin = sg.pos0 + sg.step * (128 * kt);
  const int kmax = sg.pos0 + sg.step * (128 * kt + kvalid - 1);
  const int g = p.Hq / p.Hkv;
  const uint32_t sK = base + C::kRes0, sV = base + C::kRes1;

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    const bool leader = elect_one();
    if (leader) {
      bwd_fence_maps(p, sg.chunk);
      mbar_arrive_expect_tx(bb.res_full, 2 * C::kTileBytes);
#pragma unroll
      for (int bx = 0; bx < C::kBoxes; ++bx) {
        tma_load_4d(sK + bx * C::kBoxBytes, bkmap(p, sg.chunk), bb.res_full, bx * 64, krow0, hkv, b);
        tma_load_4d(sV + bx * C::kBoxBytes, bvmap(p, sg.chunk), bb.res_full, bx * 64, krow0, hkv, b);
      }
    }
    QWalk<kDocs> w{0, g * p.n_qtiles, p.n_qtiles, hkv * g};
    int h, qt, j = 0;
    bool ok = true;
    while (ok && w.next(p, kmin, kmax, h, qt)) {
      const int st = j & 1;
      ok = warp_wait(bb.st_empty0 + 8 * st, ((j >> 1) & 1) ^ 1, bb.abort_flag, budget, kSiteBwdEmpty);
      if (!ok) break;
      const uint32_t sQ = base + C::kStage0 + st * C::kStageBytes, sDO = sQ + C::kTileBytes;
      if (leader) {
        // Q, dO and the query tile's column data (bias tiles, key windows)
        mbar_arrive_expect_tx(bb.st_full0 + 8 * st, 2 * C::kTileBytes + C::kAuxBytes);
#pragma unroll
        for (int bx = 0; bx < C::kBoxes; ++bx) {
          tma_load_4d(sQ + bx * C::kBoxBytes, &p.qmap, bb.st_full0 + 8 * st, bx * 64, 128 * qt, h, b);
          tma_load_4d(sDO + bx * C::kBoxBytes, &p.domap, bb.st_full0 + 8 * st, bx * 64, 128 * qt, h, b);
        }
        bulk_load(base + C::kAux0 + st * C::kAuxBytes,
                  p.colaux + ((int64_t(b) * p.Hq + h) * p.n_qtiles + qt) * int64_t(kColAuxBytes),
                  C::kAuxBytes, bb.st_full0 + 8 * st);
      }
      __syncwarp();
      ++j;
    }
    if (!ok) {
      // let the copies in flight land before the CTA goes away
      drain_wait(bb.res_full, 0, budget);
      for (int s = 0; s < 2; ++s) {
        const int last = (j - 1 - s) >= 0 ? ((j - 1 - s) & ~1) + s : -1;
        if (last >= 0 && last < j) drain_wait(bb.st_full0 + 8 * s, (last >> 1) & 1, budget);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA warp
    // Per pair j: S^T_j (into the S^T columns) as soon as the elementwise
    // warps have read S^T_{j-1}; then, once they have written P^T_{j-1} and
    // dS^T_{j-1} over dP^T_{j-1}, dV and dK of pair j - 1 and dP^T_j.
    const bool leader = elect_one();
    const uint32_t tS = tmem, tP = tmem + 128, tdV = tmem + 256, tdK = tmem + 384;
    bool ok = warp_wait(bb.res_full, 0, bb.abort_flag, budget, kSiteBwdKv);
    // the query tiles of this key tile, in walk order (the walk is cheap to redo)
    QWalk<kDocs> w{0, g * p.n_qtiles, p.n_qtiles, hkv * g};
    int n = 0;
    {
      QWalk<kDocs> wc{0, g * p.n_qtiles, p.n_qtiles, hkv * g};
      int hh, qq;
      while (wc.next(p, kmin, kmax, hh, qq)) ++n;
    }
    auto stage_q = [&](int jj) { return base + C::kStage0 + (jj & 1) * C::kStageBytes; };
    auto stage_b = [&](int jj) { return base + C::kAux0 + (jj & 1) * C::kAuxBytes; };
    int h, qt;
    if (ok && n > 0) {
      w.next(p, kmin, kmax, h, qt);
      ok = warp_wait(bb.st_full0, 0, bb.abort_flag, budget, kSiteBwdStage);
      if (ok) {
        tc_fence_after();
        if (leader) {
          issue_bias(tS, base + C::kOnes, stage_b(0));                      // -lse2 / c per column
          issue_abt<D>(tS, sK, stage_q(0), true);                           // S^T += K Q^T
          issue_bias(tP, base + C::kOnes, stage_b(0) + C::kBiasBytes);      // -delta per column
          issue_abt<D>(tP, sV, stage_q(0) + C::kTileBytes, true);           // dP^T += V dO^T
          mma_commit(bb.sdp_full);
        }
        __syncwarp();
      }
    }
    for (int j = 0; ok && j < n; ++j) {
      const bool more = j + 1 < n;
      const uint32_t next_full = bb.st_full0 + 8 * ((j + 1) & 1), next_par = ((j + 1) >> 1) & 1;
      bool s_next = false;  // S^T_{j+1} already issued
      if (more) {
        w.next(p, kmin, kmax, h, qt);
        ok = warp_wait(bb.s_free, j & 1, bb.abort_flag, budget, kSiteBwdSdp);
        if (!ok) break;
        // the next S^T under the elementwise work, if its stage has landed;
        // otherwise after this pair's dV, dK (which need only the elementwise
        // results)
        if (warp_phase_done(next_full, next_par)) {
          tc_fence_after();
          if (leader) {
            issue_bias(tS, base + C::kOnes, stage_b(j + 1));
            issue_abt<D>(tS, sK, stage_q(j + 1), true);
          }
          __syncwarp();
          s_next = true;
        }
      }
      ok = warp_wait(bb.ew_done, j & 1, bb.abort_flag, budget, kSiteBwdDs);
      if (!ok) break;
      tc_fence_after();
      if (leader) {
        issue_tmem_a<D>(tdV, tP, stage_q(j) + C::kTileBytes, j > 0);   // dV += P^T dO
        issue_tmem_a<D>(tdK, tP + 32, stage_q(j), j > 0);             // dK += dS^T Q
        mma_commit(bb.st_empty0 + 8 * (j & 1));
      }
      __syncwarp();
      if (more) {
        if (!s_next) {
          ok = warp_wait(next_full, next_par, bb.abort_flag, budget, kSiteBwdStage);
          if (!ok) break;
          tc_fence_after();
        }
        if (leader) {
          if (!s_next) {
            issue_bias(tS, base + C::kOnes, stage_b(j + 1));
            issue_abt<D>(tS, sK, stage_q(j + 1), true);
          }
          issue_bias(tP, base + C::kOnes, stage_b(j + 1) + C::kBiasBytes);
          issue_abt<D>(tP, sV, stage_q(j + 1) + C::kTileBytes, true);
          mma_commit(bb.sdp_full);
        }
        __syncwarp();
      }
    }
    if (leader) {
      if (ok && n > 0) mma_commit(bb.acc_full);
      mma_commit(bb.done);
    }
    __syncwarp();
    drain_wait(bb.done, 0, budget);
  } else if (warp >= 4) {
    // ---------------------------------------------------------- elementwise
    const int hw = (warp - 4) >> 2;              // column half of this warpgroup
    const int sub = warp & 3;
    const int r = sub * 32 + lane;               // key row of the tile
    const bool krow_ok = r < kvalid;
    const int kpos = sg.pos0 + sg.step * (128 * kt + r);
    const uint32_t lane_off = uint32_t(sub * 32) << 16;
    const uint32_t tS = tmem + lane_off, tP = tmem + 128 + lane_off;
    const uint32_t tdV = tmem + 256 + lane_off, tdK = tmem + 384 + lane_off;
    const float c2 = p.scale_log2;
    const uint64_t c2x2 = f2(c2, c2);
    QWalk<kDocs> w{0, g * p.n_qtiles, p.n_qtiles, hkv * g};
    int h, qt, j = 0;
    bool ok = true;
    while (ok && w.next(p, kmin, kmax, h, qt)) {
      const int st = j & 1;
      ok = warp_wait(bb.st_full0 + 8 * st, (j >> 1) & 1, bb.abort_flag, budget, kSiteBwdStage) &&
           warp_wait(bb.sdp_full, j & 1, bb.abort_flag, budget, kSiteBwdSdp);
      if (!ok) break;
      tc_fence_after();
      // the key windows of the query tile's rows (lo, hi), after the bias tiles
      const int4* awin = reinterpret_cast<const int4*>(gbase + C::kAux0 + st * C::kAuxBytes + 2 * C::kBiasBytes);
      // a mask is needed only where some key of the tile lies outside some
      // row's window (after some row's position, without documents), or
      // where the key tile is ragged
      bool masked = kvalid < 128;
      if constexpr (kDocs) {
        const int4 qw = p.qtile_pos[qt];
        masked = masked || kmax > qw.w || kmin < qw.z;
      } else {
        masked = masked || (p.causal && kmax > p.qtile_pos[qt].w);
      }
      // S^T and dP^T arrive with their column biases already added:
      // P^T = 2^(c S^T), dS^T = P^T dP^T. Both halves of this warpgroup's 64
      // columns are read first, so that S^T's columns are free for the next
      // pair's product at once; P^T and dS^T then go over dP^T's columns
      // (those this warpgroup read): P^T at [64 hw, 64 hw + 32), dS^T at
      // [64 hw + 32, 64 hw + 64), the TMEM A operands of dV and dK.
      uint32_t sv[2][32], dp[2][32];
      tmem_ld32(tS + 64 * hw, sv[0]);
      tmem_ld32(tS + 64 * hw + 32, sv[1]);
      tmem_ld32(tP + 64 * hw, dp[0]);
      tmem_ld32(tP + 64 * hw + 32, dp[1]);
      tmem_ld_wait();
      reg_fence(sv[0]);
      reg_fence(sv[1]);
      reg_fence(dp[0]);
      reg_fence(dp[1]);
      tc_fence_before();
      mbar_arrive(bb.s_free);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int i = 2 * hw + q;  // 32-column chunk of the tile
        if (masked) {
          // a score outside its column's window (or of a missing key row)
          // becomes -inf: p = 0 and dS = 0
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const int4 w = awin[(32 * i + c) / 2];  // two columns' windows
            if (!krow_ok || kpos < w.x || kpos > w.y) sv[q][c] = 0xff800000u;
            if (!krow_ok || kpos < w.z || kpos > w.w) sv[q][c + 1] = 0xff800000u;
          }
        }
        uint32_t pp[16], pd[16];
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          float x0, x1;
          f2_split(mul2(f2(__uint_as_float(sv[q][c]), __uint_as_float(sv[q][c + 1])), c2x2), x0, x1);
          const float p0 = ex2(x0), p1 = ex2(x1);
          float d0, d1;
          f2_split(mul2(f2(p0, p1), f2(__uint_as_float(dp[q][c]), __uint_as_float(dp[q][c + 1]))), d0,
                   d1);
          pp[c / 2] = pack_bf16x2(p0, p1);
          pd[c / 2] = pack_bf16x2(d0, d1);
        }
        tmem_st16(tP + 64 * hw + 16 * q, pp);
        tmem_st16(tP + 64 * hw + 32 + 16 * q, pd);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bb.ew_done);
      ++j;
    }
    // ---- epilogue: dK (times scale) and dV rows of this key tile. Each
    // thread puts its row into padded row-major tiles in shared memory, then
    // every warp stores whole rows. All eight warps reach the barrier, also
    // after an abort (the abort flag then keeps the tiles from being stored).
    const bool any = j > 0;
    if (ok && any) {
      ok = warp_wait(bb.acc_full, 0, bb.abort_flag, budget, kSiteBwdAcc);
      tc_fence_after();
    }
    float* const stK = reinterpret_cast<float*>(gbase + C::kEpiK);
    float* const stV = reinterpret_cast<float*>(gbase + C::kEpiV);
    if (ok) {
      // D / 32 column chunks, the first half of them (rounded up) to half 0
      constexpr int kNc = D / 32, kPer = (kNc + 1) / 2;
#pragma unroll 1
      for (int cc = hw * kPer; cc < min(kNc, (hw + 1) * kPer); ++cc) {
        uint32_t a[32], v[32];
        if (any) {
          tmem_ld32(tdK + 32 * cc, a);
          tmem_ld32(tdV + 32 * cc, v);
          tmem_ld_wait();
          reg_fence(a);
          reg_fence(v);
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) a[c] = v[c] = 0u;
        }
        float4* const rk = reinterpret_cast<float4*>(stK + r * C::kEpiPitch + 32 * cc);
        float4* const rv = reinterpret_cast<float4*>(stV + r * C::kEpiPitch + 32 * cc);
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          rk[c / 4] = make_float4(__uint_as_float(a[c]) * p.scale, __uint_as_float(a[c + 1]) * p.scale,
                                  __uint_as_float(a[c + 2]) * p.scale, __uint_as_float(a[c + 3]) * p.scale);
          rv[c / 4] = make_float4(__uint_as_float(v[c]), __uint_as_float(v[c + 1]),
                                  __uint_as_float(v[c + 2]), __uint_as_float(v[c + 3]));
        }
      }
    }
    named_bar_sync(1, 256);
    if (*bb.abort_flag == 0) {
      int clen;
      float *dkr, *dvr;
      if (p.ext_chunk_len != nullptr) {
        clen = __ldg(p.ext_chunk_len + sg.chunk);
        dkr = reinterpret_cast<float*>(__ldg(reinterpret_cast<const unsigned long long*>(p.ext_dk) + sg.chunk));
        dvr = reinterpret_cast<float*>(__ldg(reinterpret_cast<const unsigned long long*>(p.ext_dv) + sg.chunk));
      } else {
        clen = p.chunk_len[sg.chunk];
        dkr = p.dk[sg.chunk];
        dvr = p.dv[sg.chunk];
      }
      const int64_t row0 = (int64_t(b) * p.Hkv + hkv) * clen + krow0;
      store_staged_rows<D>(stK, dkr + row0 * D, kvalid, warp - 4, lane);
      store_staged_rows<D>(stV, dvr + row0 * D, kvalid, warp - 4, lane);
    }
  }
  bwd_teardown(tmem);
}

// ------------------------------------------------------------ dQ
// Shared memory of a dQ CTA: dO resident, rings of three K and three V tiles
// (K_j is read by S_j and, later, by dQ_j; V_j by dP_j), barriers. Q lives in
// tensor memory (the A operand of S = Q K^T), which leaves the shared memory
// for the third V tile.
template <int D>
struct DqCfg {
  static constexpr int kTileBytes = BwdCfg<D>::kTileBytes;
  static constexpr int kBoxes = BwdCfg<D>::kBoxes;
  static constexpr int kBoxBytes = BwdCfg<D>::kBoxBytes;
  static constexpr int kKSlots = 3, kVSlots = 3;
  static constexpr int kDO = 0;
  static constexpr int kK0 = kTileBytes;
  static constexpr int kV0 = kK0 + kKSlots * kTileBytes;
  static constexpr int kBar = kV0 + kVSlots * kTileBytes;
  static constexpr int kSmemBytes = kBar + 256 + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  // epilogue: dQ as a padded row-major fp32 tile over the dO and K buffers
  static constexpr int kEpiPitch = D + 4;
  static_assert(128 * kEpiPitch * 4 <= kBar, "epilogue tile fits the free buffers");
};

// One dQ CTA per (batch, query head, 128-row query tile): for every live key
// tile j, S_j = Q K_j^T and dP_j = dO V_j^T (TMEM), dS_j = P_j (dP_j - delta)
// by the elementwise warps into a TMEM region of its own, and dQ += dS_j K_j.
// The products of tile j + 1 are issued as soon as the elementwise warps have
// read S_j and dP_j, so they run while dS_j is computed; dQ_j follows.
// TMEM: S [0,128), dP [128,256), dQ [256,256+D), dS (bf16) [384,448), Q (bf16,
// written by the elementwise warps at the start) [448,448+D/2).
template <int D>
__device__ __forceinline__ void bwd_dq_tile(const BwdPlan& p, int cta) {
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  // barriers (8 bytes each): Q/dO, K ring full/empty, V ring full/empty, then
  // the single ones; the TMEM address and the abort flag after them
  constexpr int kOffK = 8, kOffV = kOffK + 16 * C::kKSlots, kOffS = kOffV + 16 * C::kVSlots;
  constexpr int kOffSlot = kOffS + 56;
  static_assert(kOffSlot + 8 <= 256, "barrier area");
  const uint32_t bars = base + C::kBar;
  const uint32_t b_res = bars, b_kfull0 = bars + kOffK, b_kempty0 = bars + kOffK + 8 * C::kKSlots,
                 b_vfull0 = bars + kOffV, b_vempty0 = bars + kOffV + 8 * C::kVSlots,
                 b_sfull = bars + kOffS, b_sdpfree = bars + kOffS + 8, b_dsfull = bars + kOffS + 16,
                 b_dsfree = bars + kOffS + 24, b_acc = bars + kOffS + 32, b_done = bars + kOffS + 40,
                 b_qready = bars + kOffS + 48;
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kBar + kOffSlot);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(gbase + C::kBar + kOffSlot + 4);
  if (threadIdx.x == 0) {
    mbar_init(b_res, 1);
    for (int i = 0; i < C::kKSlots; ++i) {
      mbar_init(b_kfull0 + 8 * i, 1);
      mbar_init(b_kempty0 + 8 * i, 1);
    }
    for (int i = 0; i < C::kVSlots; ++i) {
      mbar_init(b_vfull0 + 8 * i, 1);
      mbar_init(b_vempty0 + 8 * i, 1);
    }
    mbar_init(b_sfull, 1);
    mbar_init(b_sdpfree, 256);
    mbar_init(b_dsfull, 256);
    mbar_init(b_dsfree, 1);
    mbar_init(b_acc, 1);
    mbar_init(b_done, 1);
    mbar_init(b_qready, 256);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if ((threadIdx.x >> 5) == 1) {
    tmem_alloc(smem_addr(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned long long budget = p.timeout_ns;

  // this CTA's query tile; with a causal mask the later tiles (more keys)
  // are started first
  int u = cta;
  int qt = u % p.n_qtiles;
  if (p.causal) qt = p.n_qtiles - 1 - qt;
  u /= p.n_qtiles;
  const int hq = u % p.Hq, b = u / p.Hq;
  const int hkv = hq / (p.Hq / p.Hkv);
  // key positions some row of the tile may see: [wlo, whi]
  int wlo = 0, whi = 0x7fffffff;
  if (p.causal || p.n_docs) {
    const int4 qw = p.qtile_pos[qt];
    wlo = qw.x;
    whi = qw.y;
  }
  const uint32_t sDO = base + C::kDO;

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    const bool leader = elect_one();
    if (leader) {
      mbar_arrive_expect_tx(b_res, C::kTileBytes);
#pragma unroll
      for (int bx = 0; bx < C::kBoxes; ++bx)
        tma_load_4d(sDO + bx * C::kBoxBytes, &p.domap, b_res, bx * 64, 128 * qt, hq, b);
    }
    int jk = 0, jv = 0, fenced = -1;  // tiles whose K, V copies were issued
    bool ok = true;
    for (int k = 0; ok && k < p.n_kvsegs; ++k) {
      const KvSeg sg = bspan(p, k);
      int tb, te;
      bwd_live_tiles(p, k, wlo, whi, tb, te);
      for (int t = tb; ok && t < te; ++t) {
        const int ks = jk % C::kKSlots, vs = jv % C::kVSlots;
        ok = warp_wait(b_kempty0 + 8 * ks, ((jk / C::kKSlots) & 1) ^ 1, abort_flag, budget, kSiteBwdEmpty);
        if (!ok) break;
        if (leader) {
          if (sg.chunk != fenced) {
            bwd_fence_maps(p, sg.chunk);
            fenced = sg.chunk;
          }
          mbar_arrive_expect_tx(b_kfull0 + 8 * ks, C::kTileBytes);
#pragma unroll
          for (int bx = 0; bx < C::kBoxes; ++bx)
            tma_load_4d(base + C::kK0 + ks * C::kTileBytes + bx * C::kBoxBytes, bkmap(p, sg.chunk),
                        b_kfull0 + 8 * ks, bx * 64, sg.row0 + 128 * t, hkv, b);
        }
        ++jk;
        __syncwarp();
        ok = warp_wait(b_vempty0 + 8 * vs, ((jv / C::kVSlots) & 1) ^ 1, abort_flag, budget, kSiteBwdEmpty);
        if (!ok) break;
        if (leader) {
          mbar_arrive_expect_tx(b_vfull0 + 8 * vs, C::kTileBytes);
#pragma unroll
          for (int bx = 0; bx < C::kBoxes; ++bx)
            tma_load_4d(base + C::kV0 + vs * C::kTileBytes + bx * C::kBoxBytes, bvmap(p, sg.chunk),
                        b_vfull0 + 8 * vs, bx * 64, sg.row0 + 128 * t, hkv, b);
        }
        ++jv;
        __syncwarp();
      }
    }
    if (!ok && leader) {
      // let the copies in flight land before the CTA goes away: the last copy
      // issued into each slot
      drain_wait(b_res, 0, budget);
      for (int i = 0; i < C::kKSlots; ++i) {
        const int last = jk - 1 - ((jk - 1 - i) % C::kKSlots + C::kKSlots) % C::kKSlots;
        if (last >= 0) drain_wait(b_kfull0 + 8 * i, (last / C::kKSlots) & 1, budget);
      }
      for (int i = 0; i < C::kVSlots; ++i) {
        const int last = jv - 1 - ((jv - 1 - i) % C::kVSlots + C::kVSlots) % C::kVSlots;
        if (last >= 0) drain_wait(b_vfull0 + 8 * i, (last / C::kVSlots) & 1, budget);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA warp
    const bool leader = elect_one();
    const uint32_t tS = tmem, tP = tmem + 128, tdQ = tmem + 256, tdS = tmem + 384;
    const uint32_t tQ = tmem + 448;
    constexpr uint32_t kIdQ = idesc_bf16_f32(128, D, 0, 1);
    constexpr uint32_t kIdS = idesc_bf16_f32(128, 128, 0, 0);
    // live key tiles of this query tile
    int n = 0;
    for (int k = 0; k < p.n_kvsegs; ++k) {
      int tb, te;
      bwd_live_tiles(p, k, wlo, whi, tb, te);
      n += te - tb;
    }
    // This warp polls its barriers (never sleeps in try_wait): it then issues
    // the next products the moment their inputs are there (+2% on the 8K and
    // 32K backward; the same change in the dK/dV CTAs measured no gain).
    bool ok = warp_wait_spin(b_res, 0, abort_flag, budget, kSiteBwdKv) &&
              warp_wait_spin(b_qready, 0, abort_flag, budget, kSiteBwdKv);
    auto issue_sdp = [&](int jj) {
      const uint32_t sK = base + C::kK0 + (jj % C::kKSlots) * C::kTileBytes;
      const uint32_t sV = base + C::kV0 + (jj % C::kVSlots) * C::kTileBytes;
      // S = Q K^T: Q (bf16, two per column) is the TMEM A operand, K a K-major B
      const uint64_t kd = sdesc_sw128(sK, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_ts(tS, tQ + 8 * kk, kd + uint64_t(((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4), kIdS,
               kk > 0 ? 1u : 0u);
      issue_abt<D>(tP, sDO, sV);  // dP = dO V^T
      mma_commit(b_vempty0 + 8 * (jj % C::kVSlots));
      mma_commit(b_sfull);
    };
    if (ok && n > 0) {
      ok = warp_wait_spin(b_kfull0, 0, abort_flag, budget, kSiteBwdStage) &&
           warp_wait_spin(b_vfull0, 0, abort_flag, budget, kSiteBwdStage);
      if (ok) {
        tc_fence_after();
        if (leader) issue_sdp(0);
        __syncwarp();
      }
    }
    for (int jj = 0; ok && jj < n; ++jj) {
      if (jj + 1 < n) {
        const int j1 = jj + 1;
        ok = warp_wait_spin(b_sdpfree, jj & 1, abort_flag, budget, kSiteBwdSdp) &&
             warp_wait_spin(b_kfull0 + 8 * (j1 % C::kKSlots), (j1 / C::kKSlots) & 1, abort_flag, budget,
                       kSiteBwdStage) &&
             warp_wait_spin(b_vfull0 + 8 * (j1 % C::kVSlots), (j1 / C::kVSlots) & 1, abort_flag, budget,
                       kSiteBwdStage);
        if (!ok) break;
        tc_fence_after();
        if (leader) issue_sdp(j1);
        __syncwarp();
      }
      ok = warp_wait_spin(b_dsfull, jj & 1, abort_flag, budget, kSiteBwdDs);
      if (!ok) break;
      tc_fence_after();
      if (leader) {
        // dQ += dS K: dS (bf16) is the TMEM A operand, K_j an MN-major B
        const uint32_t sK = base + C::kK0 + (jj % C::kKSlots) * C::kTileBytes;
        const uint64_t bd = sdesc_sw128(sK, C::kBoxBytes, 1024);
#pragma unroll
        for (int kk = 0; kk < 128 / 16; ++kk)
          mma_ts(tdQ, tdS + 8 * kk, bd + uint64_t((kk * 16 * 128) >> 4), kIdQ,
                 (jj > 0 || kk > 0) ? 1u : 0u);
        mma_commit(b_dsfree);
        mma_commit(b_kempty0 + 8 * (jj % C::kKSlots));
      }
      __syncwarp();
    }
    if (leader) {
      if (ok && n > 0) mma_commit(b_acc);
      mma_commit(b_done);
    }
    __syncwarp();
    drain_wait(b_done, 0, budget);
  } else if (warp >= 4) {
    // ---------------------------------------------------------- elementwise
    const int hw = (warp - 4) >> 2;              // key-column half of this warpgroup
    const int sub = warp & 3;
    const int r = sub * 32 + lane;               // query row of the tile
    const int grow = 128 * qt + r;
    const bool rvalid = grow < p.Sq;
    const int64_t srow = (int64_t(b) * p.Hq + hq) * p.Sq + grow;
    const float lse = rvalid ? p.lse2[srow] : kInf;
    const float del = rvalid ? p.delta[srow] : 0.f;
    int rlo = 0, rhi = 0x7ffffffe;  // keys this row may see: positions [rlo, rhi]
    if (rvalid) key_window(p, bwd_row_position(p, grow), rlo, rhi);
    const uint32_t lane_off = uint32_t(sub * 32) << 16;
    const uint32_t tS = tmem + lane_off, tP = tmem + 128 + lane_off, tdQ = tmem + 256 + lane_off;
    const uint32_t tdS = tmem + 384 + lane_off;
    const uint64_t c2x2 = f2(p.scale_log2, p.scale_log2), nlse = f2(-lse, -lse), ndel = f2(-del, -del);
    {
      // this row's Q into TMEM (row = lane, two bf16 per column): warpgroup h
      // writes head-dim elements [64h, 64h + 64); rows past Sq are zero
      constexpr int kWords = D / 2 - 32 * 0;  // words of a full row
      const int w0 = 32 * hw, nw = min(32, kWords - w0);
      uint32_t qw[32];
      const uint4* src = reinterpret_cast<const uint4*>(
          p.q + int64_t(b) * p.q_sb + int64_t(hq) * p.q_sh + int64_t(grow) * p.q_sr + 2 * w0);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 v = (rvalid && 4 * i < nw) ? src[i] : make_uint4(0u, 0u, 0u, 0u);
        qw[4 * i] = v.x;
        qw[4 * i + 1] = v.y;
        qw[4 * i + 2] = v.z;
        qw[4 * i + 3] = v.w;
      }
      const uint32_t tQ = tmem + 448 + lane_off + w0;
      if (nw == 32) {
        tmem_st32(tQ, qw);
      } else if (nw == 16) {
        uint32_t h16[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) h16[i] = qw[i];
        tmem_st16(tQ, h16);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(b_qready);
    }
    int j = 0;
    bool ok = true;
    for (int k = 0; ok && k < p.n_kvsegs; ++k) {
      const KvSeg sg = bspan(p, k);
      int tb, te;
      bwd_live_tiles(p, k, wlo, whi, tb, te);
      for (int t = tb; t < te; ++t, ++j) {
        // visible keys of this row: the range [C0, L) of the key tile
        int L = min(128, sg.len - 128 * t), C0 = 0;
        if (p.causal || p.n_docs) {
          const int first = sg.pos0 + sg.step * (128 * t);
          if (sg.step == 1) {
            L = rhi < first ? 0 : min(L, rhi - first + 1);
            if (rlo > first) C0 = min(L, rlo - first);
          } else {
            L = rhi < first ? 0 : min(L, (rhi - first) / sg.step + 1);
            if (rlo > first) C0 = min(L, (rlo - first - 1) / sg.step + 1);
          }
        }
        ok = warp_wait(b_sfull, j & 1, abort_flag, budget, kSiteBwdSdp);
        if (!ok) break;
        tc_fence_after();
        uint32_t sv[2][32], dp[2][32];
        tmem_ld32(tS + 64 * hw, sv[0]);
        tmem_ld32(tS + 64 * hw + 32, sv[1]);
        tmem_ld32(tP + 64 * hw, dp[0]);
        tmem_ld32(tP + 64 * hw + 32, dp[1]);
        tmem_ld_wait();
        reg_fence(sv[0]);
        reg_fence(sv[1]);
        reg_fence(dp[0]);
        reg_fence(dp[1]);
        // S and dP are in registers: the next tile's products may overwrite them
        tc_fence_before();
        mbar_arrive(b_sdpfree);
        uint32_t pd[2][16];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int i = 2 * hw + q;
          if (L < 128 || C0 > 0) {
#pragma unroll
            for (int c = 0; c < 32; ++c)
              if (32 * i + c >= L || 32 * i + c < C0) sv[q][c] = 0xff800000u;  // -inf: p = 0
          }
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            float x0, x1;
            f2_split(fma2(f2(__uint_as_float(sv[q][c]), __uint_as_float(sv[q][c + 1])), c2x2, nlse),
                     x0, x1);
            const uint64_t pr = f2(ex2(x0), ex2(x1));
            float d0, d1;
            f2_split(mul2(pr, add2(f2(__uint_as_float(dp[q][c]), __uint_as_float(dp[q][c + 1])), ndel)),
                     d0, d1);
            pd[q][c / 2] = pack_bf16x2(d0, d1);
          }
        }
        // the previous tile's dQ product must have read its dS
        if (j > 0) {
          ok = warp_wait(b_dsfree, (j - 1) & 1, abort_flag, budget, kSiteBwdDs);
          if (!ok) break;
          tc_fence_after();
        }
        tmem_st16(tdS + 32 * hw, pd[0]);
        tmem_st16(tdS + 32 * hw + 16, pd[1]);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(b_dsfull);
      }
    }
    // ---- epilogue: dQ rows times scale, through a padded row-major tile in
    // shared memory (free once every product is complete), then whole-row
    // stores; all eight warps reach the barrier, also after an abort
    const bool any = j > 0;
    if (ok && any) {
      ok = warp_wait(b_acc, 0, abort_flag, budget, kSiteBwdAcc);
      tc_fence_after();
    }
    float* const stQ = reinterpret_cast<float*>(gbase);
    if (ok) {
      // the TMEM loads are warp-collective: every lane takes part
      constexpr int kNc = D / 32, kPer = (kNc + 1) / 2;
#pragma unroll 1
      for (int cc = hw * kPer; cc < min(kNc, (hw + 1) * kPer); ++cc) {
        uint32_t a[32];
        if (any) {
          tmem_ld32(tdQ + 32 * cc, a);
          tmem_ld_wait();
          reg_fence(a);
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) a[c] = 0u;
        }
        float4* const rq = reinterpret_cast<float4*>(stQ + r * C::kEpiPitch + 32 * cc);
#pragma unroll
        for (int c = 0; c < 32; c += 4)
          rq[c / 4] = make_float4(__uint_as_float(a[c]) * p.scale, __uint_as_float(a[c + 1]) * p.scale,
                                  __uint_as_float(a[c + 2]) * p.scale, __uint_as_float(a[c + 3]) * p.scale);
      }
    }
    named_bar_sync(1, 256);
    if (*abort_flag == 0) {
      const int nrows = min(128, p.Sq - 128 * qt);
      store_staged_rows<D>(stQ, p.dq + ((int64_t(b) * p.Hq + hq) * p.Sq + 128 * qt) * D, nrows,
                           warp - 4, lane);
    }
  }
  bwd_teardown(tmem);
}

// One launch for both: CTAs [0, n_kv_ctas) take key tiles, the rest query
// tiles. The block scheduler hands out the query-tile CTAs as the key-tile
// CTAs of the last wave retire, so neither grid leaves a partial last wave
// idle on its own.
template <int D, bool kDocs>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_kernel(const __grid_constant__ BwdPlan p,
                                                             int n_kv_ctas) {
  if (int(blockIdx.x) < n_kv_ctas)
    bwd_dkv_tile<D, kDocs>(p, int(blockIdx.x));
  else
    bwd_dq_tile<D>(p, int(blockIdx.x) - n_kv_ctas);
}

template <int D>
int launch_bwd_d(const BwdPlan& plan, const void* o, int o_fp32, int64_t o_sb, int64_t o_sh,
                 int64_t o_sr, const void* dout, const float* m, const float* l, float* lse2,
                 float* delta, int4* qtile_pos, void* stream) {
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const int64_t tiles = int64_t(plan.B) * plan.Hq * plan.n_qtiles;
  bwd_prep_kernel<D><<<unsigned(tiles), 128, 0, cs>>>(
      plan, o, o_fp32, o_sb, o_sh, o_sr, static_cast<const uint16_t*>(dout), m, l, lse2, delta,
      qtile_pos, const_cast<uint8_t*>(plan.colaux));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  constexpr int kSmem = BwdCfg<D>::kSmemBytes > DqCfg<D>::kSmemBytes ? BwdCfg<D>::kSmemBytes
                                                                    : DqCfg<D>::kSmemBytes;
  const bool docs = plan.n_docs > 0;
  auto kern = docs ? bwd_kernel<D, true> : bwd_kernel<D, false>;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem)) !=
      cudaSuccess)
    return e;
  const int64_t kv_ctas = int64_t(plan.n_ktiles) * plan.Hkv * plan.B;
  const int64_t q_ctas = int64_t(plan.n_qtiles) * plan.Hq * plan.B;
  if (kv_ctas + q_ctas > 0) {
    kern<<<unsigned(kv_ctas + q_ctas), kBwdThreads, kSmem, cs>>>(plan, int(kv_ctas));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

int launch_bwd_bf16(const BwdPlan& plan, int D, const void* o, int o_fp32, int64_t o_sb,
                    int64_t o_sh, int64_t o_sr, const void* dout, const float* m,
                    const float* l, float* lse2, float* delta, int4* qtile_pos, void* stream) {
  switch (D) {
    case 128:
      return launch_bwd_d<128>(plan, o, o_fp32, o_sb, o_sh, o_sr, dout, m, l, lse2, delta,
                               qtile_pos, stream);
    case 96:
      return launch_bwd_d<96>(plan, o, o_fp32, o_sb, o_sh, o_sr, dout, m, l, lse2, delta,
                              qtile_pos, stream);
    default:
      return launch_bwd_d<64>(plan, o, o_fp32, o_sb, o_sh, o_sr, dout, m, l, lse2, delta,
                              qtile_pos, stream);
  }
}

int read_and_clear_bwd_error(int* code) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_ra_device_error, sizeof(int));
  if (e != cudaSuccess) return e;
  *code = v;
  if (v != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_ra_device_error, &zero, sizeof(int));
  }
  return e;
}

}  // namespace ra
