// fp32 kernels on CUDA cores: the ring walk / chunk statistics in full fp32
// (no TF32, so results stay within 1e-5 of exact), and the standalone
// online-softmax merge of two sets of statistics.
//
// Sources: exercise page "systems-distributed-ring-attention-online-softmax"
// (task statement; hint 1 = max subtraction, hint 2 = the
// exp(own_max - new_max) rescale of both sides); "Ring Attention: Distributed
// Reads with Online Softmax", sections "Do not average independently
// normalized shard outputs" and "Causal masks depend on global positions".
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "ra_plan.h"

namespace ra {
namespace {

constexpr float kNegInf = -__builtin_huge_valf();
constexpr int kRows = 32;     // query rows per block
constexpr int kParts = 4;     // threads per query row (each owns head_dim / 4 lanes)
constexpr int kKeys = 32;     // keys per staged tile

__device__ __forceinline__ int find_piece(const SimtPlan& p, int row) {
  int lo = 0, hi = p.n_qpieces - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.qp[mid].row0 <= row) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// DPT = head_dim elements per thread; thread `part` owns dims part + 4*i.
template <int DPT>
__global__ void __launch_bounds__(kRows * kParts) simt_ring_kernel(const __grid_constant__ SimtPlan p) {
  constexpr int DW = DPT * kParts;  // padded head_dim
  __shared__ float sk[kKeys][DW];
  __shared__ float sv[kKeys][DW];

  const int tid = threadIdx.x;
  const int qr = tid / kParts, part = tid % kParts;
  const int bh = blockIdx.y;
  const int b = bh / p.Hq, hq = bh % p.Hq, hkv = hq / (p.Hq / p.Hkv);
  const int row0 = blockIdx.x * kRows;
  const int grow = row0 + qr;
  const bool rvalid = grow < p.Sq;
  const int D = p.D;

  // keys this row may see: positions [rlo, rhi]
  int rlo = 0, rhi = 0x7ffffffe, qseg = 0;
  {
    const int first = find_piece(p, row0);
    qseg = p.qp[first].seg;
    if (rvalid) {
      const QPiece& pc = p.qp[find_piece(p, grow)];
      key_window(p, pc.pos0 + pc.step * (grow - pc.row0), rlo, rhi);
    }
  }

  float q[DPT], o[DPT];
#pragma unroll
  for (int i = 0; i < DPT; ++i) {
    const int d = part + kParts * i;
    q[i] = (rvalid && d < D) ? p.q[int64_t(b) * p.q_sb + int64_t(hq) * p.q_sh + int64_t(grow) * p.q_sr + d] : 0.f;
    o[i] = 0.f;
  }
  float m = kNegInf, l = 0.f;

  for (int s = 0; s < p.n_chunks; ++s) {
    const int c = p.ring ? (qseg - s + p.n_chunks) % p.n_chunks : s;
    const SimtChunk& ch = p.ch[c];
    for (int k = p.chunk_seg_begin[c]; k < p.chunk_seg_begin[c + 1]; ++k) {
      const KvSeg& sg = p.ks[k];
      for (int t0 = 0; t0 < sg.len; t0 += kKeys) {
        const int nk = min(kKeys, sg.len - t0);
        __syncthreads();  // previous tile fully consumed
        for (int e = tid; e < kKeys * DW; e += kRows * kParts) {
          const int j = e / DW, d = e % DW;
          float kv = 0.f, vv = 0.f;
          if (j < nk && d < D) {
            const int64_t r = sg.row0 + t0 + j;
            kv = ch.k[int64_t(b) * ch.k_sb + int64_t(hkv) * ch.k_sh + r * ch.k_sr + d];
            vv = ch.v[int64_t(b) * ch.v_sb + int64_t(hkv) * ch.v_sh + r * ch.v_sr + d];
          }
          sk[j][d] = kv;
          sv[j][d] = vv;
        }
        __syncthreads();
        float sc[kKeys];
        float tmax = kNegInf;
#pragma unroll
        for (int j = 0; j < kKeys; ++j) {
          float acc = 0.f;
#pragma unroll
          for (int i = 0; i < DPT; ++i) acc = fmaf(q[i], sk[j][part + kParts * i], acc);
          acc += __shfl_xor_sync(0xffffffffu, acc, 1);
          acc += __shfl_xor_sync(0xffffffffu, acc, 2);
          const int kpos = sg.pos0 + sg.step * (t0 + j);
          const bool vis = j < nk && kpos >= rlo && kpos <= rhi;
          sc[j] = vis ? acc * p.scale : kNegInf;
          tmax = fmaxf(tmax, sc[j]);
        }
        const float mnew = fmaxf(m, tmax);
        if (mnew == kNegInf) continue;  // nothing visible yet
        const float alpha = (m == kNegInf) ? 0.f : expf(m - mnew);
        float lt = 0.f;
#pragma unroll
        for (int i = 0; i < DPT; ++i) o[i] *= alpha;
#pragma unroll
        for (int j = 0; j < kKeys; ++j) {
          const float w = (sc[j] == kNegInf) ? 0.f : expf(sc[j] - mnew);
          lt += w;
#pragma unroll
          for (int i = 0; i < DPT; ++i) o[i] = fmaf(w, sv[j][part + kParts * i], o[i]);
        }
        l = l * alpha + lt;
        m = mnew;
      }
    }
  }

  if (!rvalid) return;
  const int64_t orow = int64_t(b) * p.o_sb + int64_t(hq) * p.o_sh + int64_t(grow) * p.o_sr;
  const float f = p.stats_mode ? 1.f : (l > 0.f ? 1.f / l : 0.f);
#pragma unroll
  for (int i = 0; i < DPT; ++i) {
    const int d = part + kParts * i;
    if (d < D) p.out[orow + d] = o[i] * f;
  }
  if (part == 0) {
    const size_t idx = (size_t(b) * p.Hq + hq) * size_t(p.Sq) + grow;
    p.m[idx] = m;
    p.l[idx] = l;
  }
}

// ----------------------------------------------------------- merge
// One warp per row: coefficients once per row, the numerator row in 16-byte
// vectors. HBM traffic per row: read 2 * (4 D + 8) bytes, write 4 D + 8.
__device__ __forceinline__ void merge_coeffs(float m1, float m2, float& a, float& b, float& mm) {
  mm = fmaxf(m1, m2);
  a = (m1 == kNegInf) ? 0.f : expf(m1 - mm);
  b = (m2 == kNegInf) ? 0.f : expf(m2 - mm);
}

__global__ void __launch_bounds__(256) merge_vec4_kernel(int64_t rows, int D4, float4* u_acc,
                                                         float* l_acc, float* m_acc,
                                                         const float4* u_new, const float* l_new,
                                                         const float* m_new) {
  const int lane = threadIdx.x & 31;
  const int64_t w0 = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (int64_t(gridDim.x) * blockDim.x) >> 5;
  for (int64_t row = w0; row < rows; row += nw) {
    const float m1 = m_acc[row], m2 = m_new[row];
    const float l1 = l_acc[row], l2 = l_new[row];
    float a, b, mm;
    merge_coeffs(m1, m2, a, b, mm);
    float4* ua = u_acc + row * D4;
    const float4* un = u_new + row * D4;
    for (int i = lane; i < D4; i += 32) {
      const float4 x = ua[i], y = un[i];
      ua[i] = make_float4(fmaf(a, x.x, b * y.x), fmaf(a, x.y, b * y.y), fmaf(a, x.z, b * y.z),
                          fmaf(a, x.w, b * y.w));
    }
    __syncwarp();
    if (lane == 0) {
      l_acc[row] = fmaf(a, l1, b * l2);
      m_acc[row] = mm;
    }
  }
}

__global__ void __launch_bounds__(256) merge_scalar_kernel(int64_t rows, int64_t D, float* u_acc,
                                                           float* l_acc, float* m_acc,
                                                           const float* u_new, const float* l_new,
                                                           const float* m_new) {
  const int lane = threadIdx.x & 31;
  const int64_t w0 = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (int64_t(gridDim.x) * blockDim.x) >> 5;
  for (int64_t row = w0; row < rows; row += nw) {
    const float m1 = m_acc[row], m2 = m_new[row];
    const float l1 = l_acc[row], l2 = l_new[row];
    float a, b, mm;
    merge_coeffs(m1, m2, a, b, mm);
    for (int64_t i = lane; i < D; i += 32)
      u_acc[row * D + i] = fmaf(a, u_acc[row * D + i], b * u_new[row * D + i]);
    __syncwarp();
    if (lane == 0) {
      l_acc[row] = fmaf(a, l1, b * l2);
      m_acc[row] = mm;
    }
  }
}

}  // namespace

int launch_simt_f32(const SimtPlan& plan, void* stream) {
  const dim3 grid((plan.Sq + kRows - 1) / kRows, plan.B * plan.Hq);
  const dim3 block(kRows * kParts);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int dpt = (plan.D + kParts - 1) / kParts;
  if (dpt <= 1) simt_ring_kernel<1><<<grid, block, 0, st>>>(plan);
  else if (dpt <= 2) simt_ring_kernel<2><<<grid, block, 0, st>>>(plan);
  else if (dpt <= 4) simt_ring_kernel<4><<<grid, block, 0, st>>>(plan);
  else if (dpt <= 8) simt_ring_kernel<8><<<grid, block, 0, st>>>(plan);
  else if (dpt <= 16) simt_ring_kernel<16><<<grid, block, 0, st>>>(plan);
  else simt_ring_kernel<32><<<grid, block, 0, st>>>(plan);
  return cudaGetLastError();
}

// Log-sum-exp form of the merge: two normalised outputs O_a, O_b with their
// row log-sum-exps (natural log of the row's softmax denominator, in the units
// of the scaled scores). lse = log(e^lse_a + e^lse_b); O = w_a O_a + w_b O_b
// with w_x = e^(lse_x - lse). A side with lse = -inf weighs nothing; two such
// sides give O = 0, lse = -inf.
__device__ __forceinline__ void lse_coeffs(float la, float lb, float& wa, float& wb, float& ls) {
  const float mx = fmaxf(la, lb);
  if (mx == -__builtin_huge_valf()) {
    wa = wb = 0.f;
    ls = mx;
    return;
  }
  const float ea = (la == -__builtin_huge_valf()) ? 0.f : expf(la - mx);
  const float eb = (lb == -__builtin_huge_valf()) ? 0.f : expf(lb - mx);
  const float sum = ea + eb;
  wa = ea / sum;
  wb = eb / sum;
  ls = mx + logf(sum);
}

__global__ void __launch_bounds__(256) merge_lse_kernel(int64_t rows, int64_t D, float* o_acc,
                                                        float* lse_acc, const float* o_new,
                                                        const float* lse_new, int vec4) {
  const int lane = threadIdx.x & 31;
  const int64_t w0 = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (int64_t(gridDim.x) * blockDim.x) >> 5;
  for (int64_t row = w0; row < rows; row += nw) {
    float wa, wb, ls;
    lse_coeffs(lse_acc[row], lse_new[row], wa, wb, ls);
    if (vec4) {
      float4* oa = reinterpret_cast<float4*>(o_acc + row * D);
      const float4* on = reinterpret_cast<const float4*>(o_new + row * D);
      for (int64_t i = lane; i < D / 4; i += 32) {
        const float4 x = oa[i], y = on[i];
        oa[i] = make_float4(fmaf(wa, x.x, wb * y.x), fmaf(wa, x.y, wb * y.y), fmaf(wa, x.z, wb * y.z),
                            fmaf(wa, x.w, wb * y.w));
      }
    } else {
      float* oa = o_acc + row * D;
      const float* on = o_new + row * D;
      for (int64_t i = lane; i < D; i += 32) oa[i] = fmaf(wa, oa[i], wb * on[i]);
    }
    __syncwarp();
    if (lane == 0) lse_acc[row] = ls;
  }
}

// lse = m + log(l) per row, -inf where l = 0 (the row saw no key).
__global__ void __launch_bounds__(256) stats_to_lse_kernel(int64_t rows, const float* m,
                                                           const float* l, float* lse) {
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < rows;
       i += int64_t(gridDim.x) * blockDim.x)
    lse[i] = l[i] > 0.f ? m[i] + logf(l[i]) : -__builtin_huge_valf();
}

int launch_merge_lse_f32(int64_t rows, int64_t D, float* o_acc, float* lse_acc, const float* o_new,
                         const float* lse_new, int num_sms, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int64_t blocks = (rows + 7) / 8;
  const int64_t cap = int64_t(num_sms) * 16;
  if (blocks > cap) blocks = cap;
  const int vec = (D % 4 == 0) &&
                  ((reinterpret_cast<uintptr_t>(o_acc) | reinterpret_cast<uintptr_t>(o_new)) & 15u) == 0;
  merge_lse_kernel<<<unsigned(blocks), 256, 0, st>>>(rows, D, o_acc, lse_acc, o_new, lse_new, vec);
  return cudaGetLastError();
}

int launch_stats_to_lse(int64_t rows, const float* m, const float* l, float* lse, int num_sms,
                        void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int64_t blocks = (rows + 255) / 256;
  const int64_t cap = int64_t(num_sms) * 16;
  if (blocks > cap) blocks = cap;
  stats_to_lse_kernel<<<unsigned(blocks), 256, 0, st>>>(rows, m, l, lse);
  return cudaGetLastError();
}

int launch_merge_f32(int64_t rows, int64_t D, float* u_acc, float* l_acc, float* m_acc,
                     const float* u_new, const float* l_new, const float* m_new, int num_sms,
                     void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t warps_needed = rows;
  int64_t blocks = (warps_needed + 7) / 8;
  const int64_t cap = int64_t(num_sms) * 16;
  if (blocks > cap) blocks = cap;
  const bool vec = (D % 4 == 0) && ((reinterpret_cast<uintptr_t>(u_acc) | reinterpret_cast<uintptr_t>(u_new)) & 15u) == 0;
  if (vec)
    merge_vec4_kernel<<<unsigned(blocks), 256, 0, st>>>(rows, int(D / 4), reinterpret_cast<float4*>(u_acc),
                                                        l_acc, m_acc, reinterpret_cast<const float4*>(u_new),
                                                        l_new, m_new);
  else
    merge_scalar_kernel<<<unsigned(blocks), 256, 0, st>>>(rows, D, u_acc, l_acc, m_acc, u_new, l_new, m_new);
  return cudaGetLastError();
}

}  // namespace ra
