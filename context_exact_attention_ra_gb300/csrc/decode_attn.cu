// Decode over keys and values spread across c shards: split-K partials and
// their merge ("06 - Sequence / Context Parallelism", section 7: with one new
// query the attention over distributed keys needs a gather of partial
// results, like a FlashDecoding split-K).
//
// Every shard's keys are cut into pieces of kPiece local rows; one thread
// block computes the partial online-softmax state (o, m, l) of all query rows
// of one (batch, key/value head) -- the G query heads that share the head
// times the R new tokens -- over one piece, so each key and value byte is read
// from memory once.  A second kernel merges the partials of every query row
// (one block per row).  Both combine partial sums in a fixed order, so the
// results do not depend on timing.
// The work per key is 2*G*R*D multiply-adds for R*G <= 16 rows, so the path
// is bound by memory bandwidth (reading K and V once), not by arithmetic; it
// runs on the CUDA cores in fp32.
//
// Block: 8 warps.  For 32 keys at a time a warp computes the scores with one
// lane per key (q in shared memory, the lane's key row from global memory),
// takes the row maxima with shuffles, writes 2^(s - m) to shared memory, and
// then accumulates P V with one lane per 4 (D=128) or 2 (D=64) value
// columns.  The 8 warps' states are combined through shared memory at the end.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "ra_internal.h"

namespace ra {
namespace {

constexpr int kDecWarps = 8;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kDecRows = 8;      // query rows (G heads x R tokens) per block
constexpr int kPiece = 512;      // local key rows per partial

__device__ __forceinline__ long long natural_key(int r, int i, int n, int c, int layout) {
  if (layout == RA_ZIGZAG) {
    const int ch = n / 2;
    return i < ch ? static_cast<long long>(r) * ch + i : static_cast<long long>(2 * c - 1 - r) * ch + (i - ch);
  }
  if (layout == RA_STRIPED) return r + static_cast<long long>(c) * i;
  return static_cast<long long>(r) * n + i;
}

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

template <int D>
__global__ void __launch_bounds__(kDecThreads, 2)
    decode_partial_kernel(const DecodeParams p) {
  constexpr int VC = D / 32;   // value columns per lane
  __shared__ __align__(16) float qs[kDecRows][D];
  __shared__ float ps[kDecWarps][kDecRows][33];
  __shared__ float wm[kDecWarps][kDecRows];
  __shared__ float Ls[kDecRows];
  __shared__ float Os[kDecRows][D];
  __shared__ int qpos_s[kDecRows];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.Hq / p.Hkv;
  const int rows = G * p.R;                       // query rows of this (b, kv head)
  const int row_blocks = (rows + kDecRows - 1) / kDecRows;
  const int bx = blockIdx.x;
  const int rb = bx % row_blocks;
  const int g = (bx / row_blocks) % p.Hkv;
  const int b = bx / (row_blocks * p.Hkv);
  const int piece = blockIdx.y;                   // shard * pieces_per_shard + part
  const int shard = piece / p.pieces_per_shard;
  const int i0 = (piece % p.pieces_per_shard) * kPiece;
  const int i1 = min(p.n, i0 + kPiece);
  const int row0 = rb * kDecRows;
  const int nrows = min(kDecRows, rows - row0);

  // query rows: row = (head within group) * R + token
  for (int e = threadIdx.x; e < kDecRows * D; e += kDecThreads) {
    const int r = e / D, d = e % D;
    float val = 0.f;
    if (r < nrows) {
      const int rr = row0 + r;
      const int h = g * G + rr / p.R;
      const int tok = rr % p.R;
      const __nv_bfloat16* qp = static_cast<const __nv_bfloat16*>(p.q) +
                                ((static_cast<long long>(b) * p.R + tok) * p.Hq + h) * D + d;
      val = __bfloat162float(*qp) * p.scale_log2;
    }
    qs[r][d] = val;
    Os[r][d] = 0.f;
  }
  if (threadIdx.x < kDecRows) Ls[threadIdx.x] = 0.f;
  if (threadIdx.x < kDecRows) {
    const int r = threadIdx.x;
    qpos_s[r] = (r < nrows) ? p.q_pos[(row0 + r) % p.R] : INT_MIN;
  }
  __syncthreads();

  float m_run[kDecRows], l_lane[kDecRows], acc[kDecRows][VC];
#pragma unroll
  for (int r = 0; r < kDecRows; ++r) {
    m_run[r] = -INFINITY;
    l_lane[r] = 0.f;
#pragma unroll
    for (int c = 0; c < VC; ++c) acc[r][c] = 0.f;
  }

  const __nv_bfloat16* kb = static_cast<const __nv_bfloat16*>(p.k);
  const __nv_bfloat16* vb = static_cast<const __nv_bfloat16*>(p.v);
  for (int base = i0 + warp * 32; base < i1; base += kDecWarps * 32) {
    // ---- scores: lane j owns key base + j
    const int i = base + lane;
    const bool kv = i < i1;
    const long long nat = kv ? natural_key(shard, i, p.n, p.c, p.layout) : 0;
    const int kpos = static_cast<int>(nat);
    float s[kDecRows];
#pragma unroll
    for (int r = 0; r < kDecRows; ++r) s[r] = 0.f;
    if (kv) {
      const uint4* krow = reinterpret_cast<const uint4*>(kb + ((static_cast<long long>(b) * p.S + nat) * p.Hkv + g) * D);
#pragma unroll 8
      for (int c8 = 0; c8 < D / 8; ++c8) {
        const uint4 w = __ldg(krow + c8);
        const float kf[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                             bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
#pragma unroll
        for (int r = 0; r < kDecRows; ++r) {
          const float4 qa = *reinterpret_cast<const float4*>(&qs[r][c8 * 8]);
          const float4 qb = *reinterpret_cast<const float4*>(&qs[r][c8 * 8 + 4]);
          s[r] = fmaf(qa.x, kf[0], s[r]);
          s[r] = fmaf(qa.y, kf[1], s[r]);
          s[r] = fmaf(qa.z, kf[2], s[r]);
          s[r] = fmaf(qa.w, kf[3], s[r]);
          s[r] = fmaf(qb.x, kf[4], s[r]);
          s[r] = fmaf(qb.y, kf[5], s[r]);
          s[r] = fmaf(qb.z, kf[6], s[r]);
          s[r] = fmaf(qb.w, kf[7], s[r]);
        }
      }
    }
    // ---- mask, block max, probabilities
#pragma unroll
    for (int r = 0; r < kDecRows; ++r) {
      const bool vis = kv && r < nrows && (!p.causal || kpos <= qpos_s[r]);
      float sv = vis ? s[r] : -INFINITY;
      float mx = sv;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float m_new = fmaxf(m_run[r], mx);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = (m_run[r] == m_new) ? 1.f : exp2f(m_run[r] - m_new);
      const float pr = vis ? exp2f(sv - m_use) : 0.f;
      l_lane[r] = l_lane[r] * alpha + pr;
#pragma unroll
      for (int c = 0; c < VC; ++c) acc[r][c] *= alpha;
      m_run[r] = m_new;
      ps[warp][r][lane] = pr;
    }
    __syncwarp();
    // ---- P V: lane owns value columns lane*VC .. +VC-1; eight value rows
    // are loaded before any is used so their latencies overlap
    const int nk = min(32, i1 - base);
    for (int j0 = 0; j0 < nk; j0 += 8) {
      float vf[8][VC];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int j = min(j0 + u, nk - 1);
        const long long natj = natural_key(shard, base + j, p.n, p.c, p.layout);
        const __nv_bfloat16* vrow = vb + ((static_cast<long long>(b) * p.S + natj) * p.Hkv + g) * D + lane * VC;
        if constexpr (VC == 4) {
          const uint2 w = __ldg(reinterpret_cast<const uint2*>(vrow));
          vf[u][0] = bf16_lo(w.x); vf[u][1] = bf16_hi(w.x); vf[u][2] = bf16_lo(w.y); vf[u][3] = bf16_hi(w.y);
        } else {
          const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(vrow));
          vf[u][0] = bf16_lo(w); vf[u][1] = bf16_hi(w);
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (j0 + u >= nk) break;
#pragma unroll
        for (int r = 0; r < kDecRows; ++r) {
          const float pr = ps[warp][r][j0 + u];
#pragma unroll
          for (int c = 0; c < VC; ++c) acc[r][c] = fmaf(pr, vf[u][c], acc[r][c]);
        }
      }
    }
    __syncwarp();
  }

  // ---- combine the 8 warps' states into the block's partial: common max,
  // then the warps add their rescaled sums into shared memory one after the
  // other (a fixed order, so the result does not depend on timing)
  if (lane == 0) {
#pragma unroll
    for (int r = 0; r < kDecRows; ++r) wm[warp][r] = m_run[r];
  }
  __syncthreads();
  float fr[kDecRows], lr[kDecRows];
#pragma unroll
  for (int r = 0; r < kDecRows; ++r) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, wm[w][r]);
    fr[r] = (m_run[r] == -INFINITY) ? 0.f : exp2f(m_run[r] - M);
    float l = l_lane[r];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    lr[r] = l;
  }
  for (int w = 0; w < kDecWarps; ++w) {
    if (warp == w) {
#pragma unroll
      for (int r = 0; r < kDecRows; ++r) {
        if (lane == 0) Ls[r] += lr[r] * fr[r];
#pragma unroll
        for (int c = 0; c < VC; ++c) Os[r][lane * VC + c] += acc[r][c] * fr[r];
      }
    }
    __syncthreads();
  }
  for (int e = threadIdx.x; e < nrows * D; e += kDecThreads) {
    const int r = e / D, d = e % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, wm[w][r]);
    const int rr = row0 + r;
    const int h = g * G + rr / p.R;
    const int tok = rr % p.R;
    // partial layout: o [P, B, R, Hq, D]; m, l [P, B, Hq, R]
    const long long po = (((static_cast<long long>(piece) * p.B + b) * p.R + tok) * p.Hq + h) * D + d;
    p.part_o[po] = Os[r][d];
    if (d == 0) {
      const long long pm = ((static_cast<long long>(piece) * p.B + b) * p.Hq + h) * p.R + tok;
      p.part_m[pm] = M;
      p.part_l[pm] = Ls[r];
    }
  }
}

// One block of 8 warps per (b, h, token): merge the P partials, normalise,
// write out and lse.  The warps take every 8th partial; their sums are added
// in warp order.
template <int D>
__global__ void __launch_bounds__(kDecThreads) decode_merge_kernel(const DecodeParams p) {
  constexpr int VC = D / 32;
  __shared__ float red[kDecWarps];
  __shared__ float red_l[kDecWarps];
  __shared__ float red_o[kDecWarps][D];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const long long row = blockIdx.x;
  const int tok = static_cast<int>(row % p.R);
  const int h = static_cast<int>((row / p.R) % p.Hq);
  const int b = static_cast<int>(row / (static_cast<long long>(p.R) * p.Hq));
  auto mi = [&](int i) { return ((static_cast<long long>(i) * p.B + b) * p.Hq + h) * p.R + tok; };
  float M = -INFINITY;
  for (int i = threadIdx.x; i < p.P; i += kDecThreads) M = fmaxf(M, p.part_m[mi(i)]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if (lane == 0) red[warp] = M;
  __syncthreads();
  M = red[0];
#pragma unroll
  for (int w = 1; w < kDecWarps; ++w) M = fmaxf(M, red[w]);
  const float Mu = (M == -INFINITY) ? 0.f : M;
  float L = 0.f, acc[VC];
#pragma unroll
  for (int c = 0; c < VC; ++c) acc[c] = 0.f;
#pragma unroll 4
  for (int i = warp; i < p.P; i += kDecWarps) {
    const float m = p.part_m[mi(i)];
    const float f = (m == -INFINITY) ? 0.f : exp2f(m - Mu);
    L = fmaf(p.part_l[mi(i)], f, L);
    const float* po = p.part_o + (((static_cast<long long>(i) * p.B + b) * p.R + tok) * p.Hq + h) * D + lane * VC;
#pragma unroll
    for (int c = 0; c < VC; ++c) acc[c] = fmaf(po[c], f, acc[c]);
  }
  if (lane == 0) red_l[warp] = L;
#pragma unroll
  for (int c = 0; c < VC; ++c) red_o[warp][lane * VC + c] = acc[c];
  __syncthreads();
  float Lt = 0.f;
#pragma unroll
  for (int w = 0; w < kDecWarps; ++w) Lt += red_l[w];
  const float inv = (Lt > 0.f) ? 1.f / Lt : 0.f;
  const long long od = ((static_cast<long long>(b) * p.R + tok) * p.Hq + h) * D;
  for (int d = threadIdx.x; d < D; d += kDecThreads) {
    float o = 0.f;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) o += red_o[w][d];
    if (p.out_f32)
      static_cast<float*>(p.out)[od + d] = o * inv;
    else
      static_cast<__nv_bfloat16*>(p.out)[od + d] = __float2bfloat16_rn(o * inv);
  }
  if (threadIdx.x == 0 && p.lse != nullptr)
    p.lse[(static_cast<long long>(b) * p.Hq + h) * p.R + tok] =
        (Lt > 0.f) ? (M + log2f(Lt)) * 0.69314718055994531f : -INFINITY;
}

}  // namespace

int decode_pieces_per_shard(int n) { return (n + kPiece - 1) / kPiece; }
int decode_rows_per_block() { return kDecRows; }

int launch_decode(const DecodeParams& p, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int G = p.Hq / p.Hkv;
  const int row_blocks = (G * p.R + kDecRows - 1) / kDecRows;
  dim3 grid(static_cast<unsigned>(p.B * p.Hkv * row_blocks), static_cast<unsigned>(p.P));
  launch_stage() = "decode partial kernel launch";
  if (p.D == 128)
    decode_partial_kernel<128><<<grid, kDecThreads, 0, s>>>(p);
  else
    decode_partial_kernel<64><<<grid, kDecThreads, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return static_cast<int>(e);
  const unsigned rows = static_cast<unsigned>(static_cast<long long>(p.B) * p.Hq * p.R);
  launch_stage() = "decode merge kernel launch";
  if (p.D == 128)
    decode_merge_kernel<128><<<rows, kDecThreads, 0, s>>>(p);
  else
    decode_merge_kernel<64><<<rows, kDecThreads, 0, s>>>(p);
  return static_cast<int>(cudaGetLastError());
}

}  // namespace ra
