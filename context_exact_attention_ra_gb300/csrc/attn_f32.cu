// Exact fp32 blockwise attention with online softmax on the CUDA cores.
//
// The same ring walk and state update as the tensor-core kernel, in true
// fp32 (no TF32, no bf16 rounding of the probabilities), for inputs given in
// fp32.  One thread block owns one 128-row query tile of one rank and one
// query head; four threads share a query row, each holding a quarter of the
// head dimension (dimensions qtr, qtr+4, qtr+8, ...), and reduce dot products
// with two shuffles.  Keys and values are staged through shared memory 32
// keys at a time; each 32-key group is one online-softmax update:
//   m' = max(m, max_j s_j),  l' = 2^(m - m') l + sum_j 2^(s_j - m'),
//   o' = 2^(m - m') o + sum_j 2^(s_j - m') v_j          (s in base-2 units)
// ("06 - Sequence / Context Parallelism", section 4; quiz "Sequence
// Parallelism and Ring Attention", questions 3 and 7).

#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "ra_internal.h"

namespace ra {
namespace {

constexpr int kRows = 128;
constexpr int kThreadsF32 = kRows * 4;
constexpr int kSub = 32;   // keys per shared-memory stage

__device__ __forceinline__ void block_minmax(const int32_t* pos, int count, int lane, int& mn,
                                             int& mx) {
  mn = INT_MAX;
  mx = INT_MIN;
  for (int i = lane; i < count; i += 32) {
    const int p = __ldg(pos + i);
    mn = min(mn, p);
    mx = max(mx, p);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
}

template <int D>
__global__ void __launch_bounds__(kThreadsF32)
    attn_fwd_f32_kernel(const AttnParams p) {
  constexpr int DQ = D / 4;
  __shared__ float ks[kSub][D];
  __shared__ float vs[kSub][D];

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int r = tid >> 2;     // row in the tile
  const int qtr = tid & 3;    // quarter of the head dimension
  const int b = blockIdx.x / p.Hq;
  const int h = blockIdx.x % p.Hq;
  const int g = h / p.G;
  int yb = blockIdx.y;
  if (p.block_order != nullptr) yb = p.block_order[yb];
  const int rank = yb / p.q_blocks_per_rank;
  const int row0 = (yb % p.q_blocks_per_rank) * kRows;
  const int qvalid = max(0, min(kRows, p.n_q - row0));
  const int ktiles = (p.n_k + kTile - 1) / kTile;
  const long long R = static_cast<long long>(p.c) * p.n_q;
  // rows of the key/value tensors: c shards of n_k, or one gathered buffer
  const long long RK = p.kv_all ? static_cast<long long>(p.n_k) : static_cast<long long>(p.c) * p.n_k;

  const bool row_ok = r < qvalid;
  const long long qrow = static_cast<long long>(rank) * p.n_q + row0 + r;
  const int qpos = row_ok ? __ldg(p.q_pos + qrow) : INT_MIN;
  int qmn, qmx;
  block_minmax(p.q_pos + static_cast<long long>(rank) * p.n_q + row0, qvalid, lane, qmn, qmx);

  const float* qf = static_cast<const float*>(p.q);
  const float* kf = static_cast<const float*>(p.k);
  const float* vf = static_cast<const float*>(p.v);

  float q[DQ], acc[DQ];
  float m_run = -INFINITY, l_run = 0.f;
#pragma unroll
  for (int i = 0; i < DQ; ++i) {
    q[i] = row_ok ? qf[((static_cast<long long>(b) * R + qrow) * p.Hq + h) * D + qtr + 4 * i] : 0.f;
    acc[i] = 0.f;
  }
  if (p.load_state && row_ok) {
    const long long si = (static_cast<long long>(b) * p.Hq + h) * R + qrow;
    m_run = p.m_state[si];
    l_run = p.l_state[si];
    const float* so = p.o_state + ((static_cast<long long>(b) * R + qrow) * p.Hq + h) * D;
#pragma unroll
    for (int i = 0; i < DQ; ++i) acc[i] = so[qtr + 4 * i];
  }
  const float sl2 = p.scale_log2;

  for (int t = p.t_begin; t < p.t_end; ++t) {
    int src = p.kv_all ? 0 : (rank - t) % p.c;
    if (src < 0) src += p.c;
    const int32_t* kpos_src = p.k_pos + static_cast<long long>(src) * p.n_k;
    unsigned long long pairs = 0, nfull = 0, npart = 0, nskip = 0;
    for (int kt = 0; kt < ktiles; ++kt) {
      const int kvalid = min(kTile, p.n_k - kt * kTile);
      int kmn, kmx;
      block_minmax(kpos_src + kt * kTile, kvalid, lane, kmn, kmx);
      if (qvalid > 0) {
        if (!p.causal || kmx <= qmn) ++nfull;
        else if (kmn > qmx) ++nskip;
        else ++npart;
      }
      if (qvalid == 0 || (p.causal && kmn > qmx)) continue;
      for (int sub = 0; sub < kvalid; sub += kSub) {
        const int nk = min(kSub, kvalid - sub);
        __syncthreads();
        for (int e = tid; e < kSub * D; e += kThreadsF32) {
          const int kk = e / D, d = e % D;
          float kv = 0.f, vv = 0.f;
          if (kk < nk) {
            const long long krow = static_cast<long long>(p.kv_by_holder ? rank : src) * p.n_k +
                                   kt * kTile + sub + kk;
            const long long off = ((static_cast<long long>(b) * RK + krow) * p.Hkv + g) * D + d;
            kv = kf[off];
            vv = vf[off];
          }
          ks[kk][d] = kv;
          vs[kk][d] = vv;
        }
        __syncthreads();
        float s[kSub];
        float mx = -INFINITY;
#pragma unroll
        for (int kk = 0; kk < kSub; ++kk) {
          float part = 0.f;
#pragma unroll
          for (int i = 0; i < DQ; ++i) part = fmaf(q[i], ks[kk][qtr + 4 * i], part);
          part += __shfl_xor_sync(0xffffffffu, part, 1);
          part += __shfl_xor_sync(0xffffffffu, part, 2);
          bool vis = kk < nk;
          if (vis && p.causal) vis = __ldg(kpos_src + kt * kTile + sub + kk) <= qpos;
          s[kk] = vis ? part * sl2 : -INFINITY;
          mx = fmaxf(mx, s[kk]);
          pairs += (vis && row_ok && qtr == 0) ? 1ull : 0ull;
        }
        const float m_new = fmaxf(m_run, mx);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = (m_run == m_new) ? 1.f : exp2f(m_run - m_new);
        float sum = 0.f;
#pragma unroll
        for (int i = 0; i < DQ; ++i) acc[i] *= alpha;
#pragma unroll
        for (int kk = 0; kk < kSub; ++kk) {
          const float pk = (s[kk] == -INFINITY) ? 0.f : exp2f(s[kk] - m_use);
          sum += pk;
#pragma unroll
          for (int i = 0; i < DQ; ++i) acc[i] = fmaf(pk, vs[kk][qtr + 4 * i], acc[i]);
        }
        l_run = l_run * alpha + sum;
        m_run = m_new;
      }
    }
    if (p.work != nullptr) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) pairs += __shfl_xor_sync(0xffffffffu, pairs, o);
      ra_work* w = p.work + static_cast<long long>(rank) * p.c + t;
      if (lane == 0 && pairs > 0) atomicAdd(reinterpret_cast<unsigned long long*>(&w->pairs), pairs);
      if (tid == 0) {
        atomicAdd(reinterpret_cast<unsigned long long*>(&w->tiles_full), nfull);
        atomicAdd(reinterpret_cast<unsigned long long*>(&w->tiles_partial), npart);
        atomicAdd(reinterpret_cast<unsigned long long*>(&w->tiles_skipped), nskip);
      }
    }
  }

  if (!row_ok) return;
  if (p.finalize) {
    const int orow = qpos;
    const float inv_l = (l_run > 0.f) ? 1.f / l_run : 0.f;
    float* dst = static_cast<float*>(p.out) + ((static_cast<long long>(b) * p.S_out + orow) * p.Hq + h) * D;
#pragma unroll
    for (int i = 0; i < DQ; ++i) dst[qtr + 4 * i] = acc[i] * inv_l;
    if (qtr == 0 && p.lse != nullptr)
      p.lse[(static_cast<long long>(b) * p.Hq + h) * p.S_out + orow] =
          (l_run > 0.f) ? (m_run + log2f(l_run)) * 0.69314718055994531f : -INFINITY;
  }
  if (p.store_state) {
    float* so = p.o_state + ((static_cast<long long>(b) * R + qrow) * p.Hq + h) * D;
#pragma unroll
    for (int i = 0; i < DQ; ++i) so[qtr + 4 * i] = acc[i];
    if (qtr == 0) {
      const long long si = (static_cast<long long>(b) * p.Hq + h) * R + qrow;
      p.m_state[si] = m_run;
      p.l_state[si] = l_run;
    }
  }
}

}  // namespace

int launch_attn_f32(const AttnParams& p, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  dim3 grid(static_cast<unsigned>(p.B * p.Hq), static_cast<unsigned>(p.c * p.q_blocks_per_rank));
  if (p.D == 64)
    attn_fwd_f32_kernel<64><<<grid, kThreadsF32, 0, s>>>(p);
  else if (p.D == 128)
    attn_fwd_f32_kernel<128><<<grid, kThreadsF32, 0, s>>>(p);
  else
    return static_cast<int>(cudaErrorInvalidValue);
  return static_cast<int>(cudaGetLastError());
}

}  // namespace ra
