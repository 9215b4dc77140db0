// Bandwidth-bound kernels around the attention kernels: state
// initialisation, the shard pack of a ring call, the log-sum-exp merge of
// partial states, the heavy-first block order, and the device error word.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <mutex>

#include "ra_internal.h"

namespace ra {
namespace {

// The device error word (index 0) and, at byte offset 8, the device address
// of its host mirror (null until the host registers one).
__device__ __align__(16) unsigned int g_error_block[4] = {0u, 0u, 0u, 0u};

__global__ void state_init_kernel(long long n_o, long long n_ml, float* o, float* m, float* l) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n_o / 4;
       i += stride)
    reinterpret_cast<float4*>(o)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n_ml;
       i += stride) {
    m[i] = -INFINITY;
    l[i] = 0.f;
  }
}

__global__ void zero_kernel(uint4* p, long long n16) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n16;
       i += stride)
    p[i] = make_uint4(0u, 0u, 0u, 0u);
}

// Natural row of local row `i` of rank `r` (contiguous: [r n, (r+1) n);
// zig-zag: chunks r and 2c-1-r of length n/2; striped: r + c i).
__device__ __forceinline__ int natural_row(int r, int i, int n, int c, int layout) {
  if (layout == RA_ZIGZAG) {
    const int ch = n / 2;
    return i < ch ? r * ch + i : (2 * c - 1 - r) * ch + (i - ch);
  }
  if (layout == RA_STRIPED) return r + c * i;
  return r * n + i;
}

// One block per (packed row, batch): copies the row's q, k and v heads.
__global__ void pack_kernel(const uint4* q, const uint4* k, const uint4* v, int S, int n, int c,
                            int layout, int q_vec, int kv_vec, uint4* qp, uint4* kp, uint4* vp,
                            int32_t* pos) {
  const int row = blockIdx.x;
  const int b = blockIdx.y;
  const int nat = natural_row(row / n, row % n, n, c, layout);
  if (q != nullptr) {   // null: K, V and positions only (Q is copied separately)
    const long long qs = (static_cast<long long>(b) * S + nat) * q_vec;
    const long long qd = (static_cast<long long>(b) * S + row) * q_vec;
    for (int i = threadIdx.x; i < q_vec; i += blockDim.x) qp[qd + i] = q[qs + i];
  }
  const long long ks = (static_cast<long long>(b) * S + nat) * kv_vec;
  const long long kd = (static_cast<long long>(b) * S + row) * kv_vec;
  for (int i = threadIdx.x; i < kv_vec; i += blockDim.x) {
    kp[kd + i] = k[ks + i];
    vp[kd + i] = v[ks + i];
  }
  if (b == 0 && threadIdx.x == 0) pos[row] = nat;
}

// Heavy-first order of the query blocks of a causal ring: a block's key is
// the largest position among its rows; blocks are listed by key, descending
// (ties by index), so the longest causal rows start first.  With per_rank the
// blocks of each rank are ordered among themselves, rank r's list at
// order[r * blocks_per_rank ...].  One thread block: each warp reduces the
// keys of a share of the blocks (lanes over rows), keys live in shared memory.
__global__ void block_order_kernel(const int32_t* pos, int c, int n, int rows_per_block,
                                   int blocks_per_rank, int per_rank, int32_t* order) {
  extern __shared__ int keys[];
  const int total = c * blocks_per_rank;
  const int lane = threadIdx.x & 31;
  for (int y = threadIdx.x >> 5; y < total; y += blockDim.x >> 5) {
    const int r = y / blocks_per_rank;
    const int i0 = (y % blocks_per_rank) * rows_per_block;
    const int i1 = min(n, i0 + rows_per_block);
    int mx = INT_MIN;
    for (int i = i0 + lane; i < i1; i += 32) mx = max(mx, pos[static_cast<long long>(r) * n + i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) keys[y] = mx;
  }
  __syncthreads();
  for (int y = threadIdx.x; y < total; y += blockDim.x) {
    const int ky = keys[y];
    const int o0 = per_rank ? (y / blocks_per_rank) * blocks_per_rank : 0;
    const int o1 = per_rank ? o0 + blocks_per_rank : total;
    int before = 0;
    for (int o = o0; o < o1; ++o) {
      const int ko = keys[o];
      before += (ko > ky || (ko == ky && o < y)) ? 1 : 0;
    }
    order[o0 + before] = y;
  }
}

__global__ void tile_range_kernel(const int32_t* pos, int c, int n, int tiles, int2* out) {
  const long long warp_id = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp_id >= static_cast<long long>(c) * tiles) return;
  const int r = static_cast<int>(warp_id / tiles);
  const int t = static_cast<int>(warp_id % tiles);
  const int a = t * kTile;
  const int e = min(n, a + kTile);
  int mn = INT_MAX, mx = INT_MIN;
  for (int i = a + lane; i < e; i += 32) {
    const int v = pos[static_cast<long long>(r) * n + i];
    mn = min(mn, v);
    mx = max(mx, v);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  if (lane == 0) out[warp_id] = make_int2(mn, mx);
}

struct MergeParams {
  MergeArgs a;
  int B, S, Hq, D, out_dtype, S_out;
  void* out;
  float* lse;
  const int32_t* out_row;
};

// One warp per kMergeRows rows of (b, s, h), h fastest -- the order of the
// partial outputs in memory, so a warp reads one contiguous stretch and
// neighbouring warps the next ones; lanes hold D/32 consecutive columns of
// each row.  Two passes: first every partial's m and l (one lane per
// (partial, row) pair) give the row maximum M = max_p m_p, the weights
// w_p = 2^(m_p - M) and L = sum_p w_p l_p (base-2 units); then the o rows are
// summed, acc = sum_p w_p o_p, with the next partial's loads issued before the
// current one is added -- no exponential between two partials' loads.
// out = acc / L, lse = ln 2 (M + log2 L).
constexpr int kMergeRows = 4;

template <int D>
__global__ void __launch_bounds__(256, 4) merge_kernel(const MergeParams mp) {
  constexpr int V = D / 32;   // floats per lane
  constexpr int R = kMergeRows;
  constexpr int PC = 32 / R;  // partials whose weights one pass of the lanes covers
  const long long warp_id = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const long long rows = static_cast<long long>(mp.B) * mp.Hq * mp.S;
  const long long row0 = warp_id * R;
  if (row0 >= rows) return;
  // lane = pl * R + r holds partial (p0 + pl) of row r: (b, s, h) of row r and
  // the index of its m and l in [B, Hq, S]
  const int my_r = lane % R;
  const int my_pl = lane / R;
  const long long my_row = min(row0 + my_r, rows - 1);
  const long long q0 = my_row / mp.Hq;
  const int my_h = static_cast<int>(my_row - q0 * mp.Hq);
  const int my_s = static_cast<int>(q0 % mp.S);
  const int my_b = static_cast<int>(q0 / mp.S);
  const long long my_si = (static_cast<long long>(my_b) * mp.Hq + my_h) * mp.S + my_s;
  const long long obase = row0 * D + lane * V;   // o is [B, S, Hq, D]: these rows are consecutive
  const int nlive = static_cast<int>(min(static_cast<long long>(R), rows - row0));
  const int P = mp.a.P;

  // pass 1: row maximum over the partials (lanes of one row: lane % R equal)
  float Mx = -INFINITY;
  for (int p0 = 0; p0 < P; p0 += PC) {
    const int p = p0 + my_pl;
    if (p < P) Mx = fmaxf(Mx, __ldg(mp.a.ms[p] + my_si));
  }
#pragma unroll
  for (int o = R; o < 32; o <<= 1) Mx = fmaxf(Mx, __shfl_xor_sync(0xffffffffu, Mx, o));

  float acc[R][V];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int i = 0; i < V; ++i) acc[r][i] = 0.f;
  float Lsum = 0.f;   // this lane's share of L for row my_r
  auto load = [&](int p, float (&o_)[R][V]) {
    const float* opp = mp.a.outs[p] + obase;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (r < nlive) {
        if constexpr (V == 4) {
          const float4 f = __ldcs(reinterpret_cast<const float4*>(opp + r * D));
          o_[r][0] = f.x; o_[r][1] = f.y; o_[r][2] = f.z; o_[r][3] = f.w;
        } else {
          const float2 f = __ldcs(reinterpret_cast<const float2*>(opp + r * D));
          o_[r][0] = f.x; o_[r][1] = f.y;
        }
      } else {
#pragma unroll
        for (int i = 0; i < V; ++i) o_[r][i] = 0.f;
      }
    }
  };
  float ov[R][V];
  load(0, ov);
  for (int p0 = 0; p0 < P; p0 += PC) {
    // pass 2 for partials p0 .. p0 + PC - 1: this lane's weight and its share of L
    const int pw = p0 + my_pl;
    float w = 0.f;
    if (pw < P) {
      const float mv = __ldg(mp.a.ms[pw] + my_si);
      w = (mv == -INFINITY) ? 0.f : exp2f(mv - Mx);
      Lsum = fmaf(__ldg(mp.a.ls[pw] + my_si), w, Lsum);
    }
    const int pend = min(P, p0 + PC);
    for (int p = p0; p < pend; ++p) {
      float on[R][V];
      if (p + 1 < P) load(p + 1, on);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float wr = __shfl_sync(0xffffffffu, w, (p - p0) * R + r);
#pragma unroll
        for (int i = 0; i < V; ++i) acc[r][i] = fmaf(ov[r][i], wr, acc[r][i]);
      }
      if (p + 1 < P) {
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int i = 0; i < V; ++i) ov[r][i] = on[r][i];
      }
    }
  }
#pragma unroll
  for (int o = R; o < 32; o <<= 1) Lsum += __shfl_xor_sync(0xffffffffu, Lsum, o);
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const float L = __shfl_sync(0xffffffffu, Lsum, r);
    const float M = __shfl_sync(0xffffffffu, Mx, r);
    const int hh = __shfl_sync(0xffffffffu, my_h, r);
    const int ss = __shfl_sync(0xffffffffu, my_s, r);
    const int bb = __shfl_sync(0xffffffffu, my_b, r);
    if (r >= nlive) continue;
    const float inv = (L > 0.f) ? 1.f / L : 0.f;
    const int orow = (mp.out_row != nullptr) ? mp.out_row[ss] : ss;
    const long long od = ((static_cast<long long>(bb) * mp.S_out + orow) * mp.Hq + hh) * D + lane * V;
    if (mp.out_dtype == RA_F32) {
      float* o = static_cast<float*>(mp.out) + od;
      if constexpr (V == 4)
        *reinterpret_cast<float4*>(o) =
            make_float4(acc[r][0] * inv, acc[r][1] * inv, acc[r][2] * inv, acc[r][3] * inv);
      else
        *reinterpret_cast<float2*>(o) = make_float2(acc[r][0] * inv, acc[r][1] * inv);
    } else {
      __nv_bfloat16* o = static_cast<__nv_bfloat16*>(mp.out) + od;
      if constexpr (V == 4) {
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc[r][0] * inv, acc[r][1] * inv);
        __nv_bfloat162 hi = __floats2bfloat162_rn(acc[r][2] * inv, acc[r][3] * inv);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t*>(&lo);
        u.y = *reinterpret_cast<uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(o) = u;
      } else {
        *reinterpret_cast<__nv_bfloat162*>(o) = __floats2bfloat162_rn(acc[r][0] * inv, acc[r][1] * inv);
      }
    }
    if (lane == 0 && mp.lse != nullptr)
      mp.lse[(static_cast<long long>(bb) * mp.Hq + hh) * mp.S_out + orow] =
          (L > 0.f) ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
  }
}

// Two to four partials: one warp per few_rows(P) rows, every load of the warp --
// each partial's o rows, and its m and l (one lane per (partial, row) pair) --
// issued before any of them is used, so a warp waits for memory once.  Then
// per row M = max_p m_p, w_p = 2^(m_p - M) (one lane each), L = sum_p w_p l_p
// and out = sum_p w_p o_p / L, lse = ln 2 (M + log2 L): the same sums as
// merge_kernel, in the same order over the partials.
// rows per warp: four (two for four partials, to stay within 64 registers)
__host__ __device__ constexpr int few_rows(int P) { return P == 4 ? 2 : 4; }

template <int D, int P>
__global__ void __launch_bounds__(256, 4) merge_few_kernel(const MergeParams mp) {
  constexpr int V = D / 32;   // floats per lane
  constexpr int R = few_rows(P);
  static_assert(P * R <= 32, "one lane per (partial, row) pair");
  const long long warp_id = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const long long rows = static_cast<long long>(mp.B) * mp.Hq * mp.S;
  const long long row0 = warp_id * R;
  if (row0 >= rows) return;
  const int nlive = static_cast<int>(min(static_cast<long long>(R), rows - row0));
  // o is [B, S, Hq, D]: the warp's rows are consecutive
  float o[P][R][V];
#pragma unroll
  for (int p = 0; p < P; ++p) {
    const float* opp = mp.a.outs[p] + row0 * D + lane * V;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (r < nlive) {
        if constexpr (V == 4) {
          const float4 f = __ldcs(reinterpret_cast<const float4*>(opp + r * D));
          o[p][r][0] = f.x; o[p][r][1] = f.y; o[p][r][2] = f.z; o[p][r][3] = f.w;
        } else {
          const float2 f = __ldcs(reinterpret_cast<const float2*>(opp + r * D));
          o[p][r][0] = f.x; o[p][r][1] = f.y;
        }
      } else {
#pragma unroll
        for (int i = 0; i < V; ++i) o[p][r][i] = 0.f;
      }
    }
  }
  // lane k = p * R + r: m and l of partial p for row r, in [B, Hq, S]
  const int kp = lane / R, kr = lane % R;
  const long long krow = min(row0 + kr, rows - 1);
  const long long q0 = krow / mp.Hq;
  const int k_h = static_cast<int>(krow - q0 * mp.Hq);
  const int k_s = static_cast<int>(q0 % mp.S);
  const int k_b = static_cast<int>(q0 / mp.S);
  float mk = -INFINITY, lk = 0.f;
  if (kp < P && kr < nlive) {
    const long long si = (static_cast<long long>(k_b) * mp.Hq + k_h) * mp.S + k_s;
    mk = __ldg(mp.a.ms[kp] + si);
    lk = __ldg(mp.a.ls[kp] + si);
  }
  // this lane's row maximum and weight
  float Mk = -INFINITY;
#pragma unroll
  for (int p = 0; p < P; ++p) Mk = fmaxf(Mk, __shfl_sync(0xffffffffu, mk, p * R + kr));
  const float wk = (mk == -INFINITY) ? 0.f : exp2f(mk - Mk);
  const float lw = lk * wk;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    float acc[V];
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = 0.f;
    float L = 0.f;
#pragma unroll
    for (int p = 0; p < P; ++p) {
      const float w = __shfl_sync(0xffffffffu, wk, p * R + r);
      L += __shfl_sync(0xffffffffu, lw, p * R + r);
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] = fmaf(o[p][r][i], w, acc[i]);
    }
    const float M = __shfl_sync(0xffffffffu, Mk, r);
    const int hh = __shfl_sync(0xffffffffu, k_h, r);
    const int ss = __shfl_sync(0xffffffffu, k_s, r);
    const int bb = __shfl_sync(0xffffffffu, k_b, r);
    if (r >= nlive) continue;
    const float inv = (L > 0.f) ? 1.f / L : 0.f;
    const int orow = (mp.out_row != nullptr) ? mp.out_row[ss] : ss;
    const long long od = ((static_cast<long long>(bb) * mp.S_out + orow) * mp.Hq + hh) * D + lane * V;
    if (mp.out_dtype == RA_F32) {
      float* op = static_cast<float*>(mp.out) + od;
      if constexpr (V == 4)
        *reinterpret_cast<float4*>(op) = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
      else
        *reinterpret_cast<float2*>(op) = make_float2(acc[0] * inv, acc[1] * inv);
    } else {
      __nv_bfloat16* op = static_cast<__nv_bfloat16*>(mp.out) + od;
      if constexpr (V == 4) {
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
        __nv_bfloat162 hi = __floats2bfloat162_rn(acc[2] * inv, acc[3] * inv);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t*>(&lo);
        u.y = *reinterpret_cast<uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(op) = u;
      } else {
        *reinterpret_cast<__nv_bfloat162*>(op) = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
      }
    }
    if (lane == 0 && mp.lse != nullptr)
      mp.lse[(static_cast<long long>(bb) * mp.Hq + hh) * mp.S_out + orow] =
          (L > 0.f) ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
  }
}

// One partial (the per-step mode's last step): out = o / l and
// lse = m + log2 l, with m in base-2 units -- the fused kernel's epilogue
// arithmetic, so both modes agree bit for bit.  Each thread owns one 16-byte
// slice of kFinRows consecutive rows ((b, s, h) with h fastest, the order of o
// in memory) and issues all their loads before using any; a row's m and l are
// fetched once per group of lanes, which leaves eight rows (128 bytes of loads
// per thread) within 64 registers, four blocks per SM.
constexpr int kFinRows = 8;

template <int D>
__global__ void __launch_bounds__(256, 4) finalize_kernel(const MergeParams mp) {
  constexpr int C = D / 4;   // float4 slices per row: the lanes of a group
  static_assert(2 * kFinRows <= C, "m and l of a group's rows are fetched by its first 2 kFinRows lanes");
  const long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  const long long rows = static_cast<long long>(mp.B) * mp.Hq * mp.S;
  const int c4 = static_cast<int>(t % C);
  const long long row0 = (t / C) * kFinRows;
  if (row0 >= rows) return;   // whole groups of C lanes leave together
  const float* o = mp.a.outs[0];
  // lane c4 < kFinRows owns row row0 + c4: its (b, s, h) and its m; lane
  // kFinRows + c4 the same row's l; the values reach the group by shuffles
  const long long my_row = min(row0 + (c4 % kFinRows), rows - 1);
  const long long q0 = my_row / mp.Hq;
  const int my_h = static_cast<int>(my_row - q0 * mp.Hq);
  const int my_s = static_cast<int>(q0 % mp.S);
  const int my_b = static_cast<int>(q0 / mp.S);
  const long long my_si = (static_cast<long long>(my_b) * mp.Hq + my_h) * mp.S + my_s;
  const float ml = (c4 < 2 * kFinRows) ? (c4 < kFinRows ? mp.a.ms[0] : mp.a.ls[0])[my_si] : 0.f;
  float4 ov[kFinRows];
#pragma unroll
  for (int r = 0; r < kFinRows; ++r)
    ov[r] = (row0 + r < rows) ? __ldcs(reinterpret_cast<const float4*>(o + (row0 + r) * D) + c4)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
  const unsigned gmask = (C == 32) ? 0xffffffffu : (0xffffu << (threadIdx.x & 16));
#pragma unroll
  for (int r = 0; r < kFinRows; ++r) {
    const float mv = __shfl_sync(gmask, ml, r, C);
    const float lv = __shfl_sync(gmask, ml, kFinRows + r, C);
    const int hh = __shfl_sync(gmask, my_h, r, C);
    const int ss = __shfl_sync(gmask, my_s, r, C);
    const int bb = __shfl_sync(gmask, my_b, r, C);
    if (row0 + r >= rows) break;
    const float inv = (lv > 0.f) ? 1.f / lv : 0.f;
    const int orow = (mp.out_row != nullptr) ? mp.out_row[ss] : ss;
    const long long od = ((static_cast<long long>(bb) * mp.S_out + orow) * mp.Hq + hh) * D + c4 * 4;
    if (mp.out_dtype == RA_F32) {
      *reinterpret_cast<float4*>(static_cast<float*>(mp.out) + od) =
          make_float4(ov[r].x * inv, ov[r].y * inv, ov[r].z * inv, ov[r].w * inv);
    } else {
      __nv_bfloat162 lo = __floats2bfloat162_rn(ov[r].x * inv, ov[r].y * inv);
      __nv_bfloat162 hi = __floats2bfloat162_rn(ov[r].z * inv, ov[r].w * inv);
      uint2 w;
      w.x = *reinterpret_cast<uint32_t*>(&lo);
      w.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(mp.out) + od) = w;
    }
    if (c4 == 0 && mp.lse != nullptr)
      mp.lse[(static_cast<long long>(bb) * mp.Hq + hh) * mp.S_out + orow] =
          (lv > 0.f) ? (mv + log2f(lv)) * 0.69314718055994531f : -INFINITY;
  }
}

int grid_for(long long work, int threads) {
  long long blocks = (work + threads - 1) / threads;
  if (blocks < 1) blocks = 1;
  if (blocks > 152LL * 32) blocks = 152LL * 32;   // grid-stride beyond 32 waves of 152 SMs
  return static_cast<int>(blocks);
}

}  // namespace

int launch_state_init(int B, int rows, int Hq, int D, float* o, float* m, float* l, void* stream) {
  const long long n_o = static_cast<long long>(B) * rows * Hq * D;
  const long long n_ml = static_cast<long long>(B) * Hq * rows;
  if (n_o == 0) return 0;
  state_init_kernel<<<grid_for(n_o / 4, 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      n_o, n_ml, o, m, l);
  return static_cast<int>(cudaGetLastError());
}

int launch_zero(void* ptr, size_t bytes, void* stream) {
  if (bytes == 0) return 0;
  const long long n16 = static_cast<long long>(bytes / 16);
  zero_kernel<<<grid_for(n16, 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint4*>(ptr), n16);
  return static_cast<int>(cudaGetLastError());
}

int launch_pack(const void* q, const void* k, const void* v, int B, int S, int Hq, int Hkv, int D,
                int elem_bytes, int c, int layout, void* qp, void* kp, void* vp, int32_t* pos,
                void* stream) {
  if (S == 0 || B == 0) return 0;
  const int n = S / c;
  const int q_vec = Hq * D * elem_bytes / 16;
  const int kv_vec = Hkv * D * elem_bytes / 16;
  dim3 grid(static_cast<unsigned>(S), static_cast<unsigned>(B));
  pack_kernel<<<grid, 128, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(q), static_cast<const uint4*>(k), static_cast<const uint4*>(v), S,
      n, c, layout, q_vec, kv_vec, static_cast<uint4*>(qp), static_cast<uint4*>(kp),
      static_cast<uint4*>(vp), pos);
  return static_cast<int>(cudaGetLastError());
}

int launch_tile_ranges(const int32_t* pos, int c, int n, int2* ranges, void* stream) {
  const int tiles = (n + kTile - 1) / kTile;
  const long long warps = static_cast<long long>(c) * tiles;
  if (warps == 0) return 0;
  tile_range_kernel<<<static_cast<unsigned>((warps * 32 + 255) / 256), 256, 0,
                      static_cast<cudaStream_t>(stream)>>>(pos, c, n, tiles, ranges);
  return static_cast<int>(cudaGetLastError());
}

int launch_block_order(const int32_t* pos, int c, int n, int rows_per_block, int blocks_per_rank,
                       int32_t* order, void* stream, int per_rank) {
  const int total = c * blocks_per_rank;
  if (total == 0) return 0;
  if (total > kMaxOrderedBlocks) return static_cast<int>(cudaErrorInvalidValue);
  block_order_kernel<<<1, 1024, total * sizeof(int), static_cast<cudaStream_t>(stream)>>>(
      pos, c, n, rows_per_block, blocks_per_rank, per_rank, order);
  return static_cast<int>(cudaGetLastError());
}

int launch_merge(const MergeArgs& a, int B, int S, int Hq, int D, int out_dtype, void* out,
                 float* lse, const int32_t* out_row, int S_out, void* stream) {
  const long long rows = static_cast<long long>(B) * Hq * S;
  if (rows == 0) return 0;
  MergeParams mp;
  mp.a = a;
  mp.B = B;
  mp.S = S;
  mp.Hq = Hq;
  mp.D = D;
  mp.out_dtype = out_dtype;
  mp.S_out = S_out;
  mp.out = out;
  mp.lse = lse;
  mp.out_row = out_row;
  const int threads = 256;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (a.P == 1) {
    const long long nthreads = (rows + kFinRows - 1) / kFinRows * (D / 4);
    const long long fblocks = (nthreads + threads - 1) / threads;
    if (D == 128)
      finalize_kernel<128><<<static_cast<unsigned>(fblocks), threads, 0, s>>>(mp);
    else if (D == 64)
      finalize_kernel<64><<<static_cast<unsigned>(fblocks), threads, 0, s>>>(mp);
    else
      return static_cast<int>(cudaErrorInvalidValue);
    return static_cast<int>(cudaGetLastError());
  }
  if (a.P <= 4 && (D == 128 || D == 64)) {
    const long long fwarps = (rows + few_rows(a.P) - 1) / few_rows(a.P);
    const unsigned fblocks = static_cast<unsigned>((fwarps * 32 + threads - 1) / threads);
    if (D == 128) {
      if (a.P == 2) merge_few_kernel<128, 2><<<fblocks, threads, 0, s>>>(mp);
      else if (a.P == 3) merge_few_kernel<128, 3><<<fblocks, threads, 0, s>>>(mp);
      else merge_few_kernel<128, 4><<<fblocks, threads, 0, s>>>(mp);
    } else {
      if (a.P == 2) merge_few_kernel<64, 2><<<fblocks, threads, 0, s>>>(mp);
      else if (a.P == 3) merge_few_kernel<64, 3><<<fblocks, threads, 0, s>>>(mp);
      else merge_few_kernel<64, 4><<<fblocks, threads, 0, s>>>(mp);
    }
    return static_cast<int>(cudaGetLastError());
  }
  const long long warps = (rows + kMergeRows - 1) / kMergeRows;
  const long long blocks = (warps * 32 + threads - 1) / threads;
  if (D == 128)
    merge_kernel<128><<<static_cast<unsigned>(blocks), threads, 0, s>>>(mp);
  else if (D == 64)
    merge_kernel<64><<<static_cast<unsigned>(blocks), threads, 0, s>>>(mp);
  else
    return static_cast<int>(cudaErrorInvalidValue);
  return static_cast<int>(cudaGetLastError());
}

const char*& launch_stage() {
  thread_local const char* stage = "kernel launch";
  return stage;
}

namespace {
// Host mirrors of the device error words: one 64-byte slot per device in one
// page of this library's own memory, registered (pinned and mapped into every
// device's address space) on first use.  The library allocates nothing for it.
constexpr int kMaxDevices = 64;
alignas(4096) unsigned int g_mirror_page[kMaxDevices * 16];

struct ErrorHandles {
  unsigned long long ctx = 0;
  unsigned int* word = nullptr;
  volatile unsigned int* mirror = nullptr;   // host view, or null
};

std::mutex g_error_mu;
ErrorHandles g_error_cache[kMaxDevices];
bool g_mirror_registered = false;
bool g_mirror_failed = false;
}  // namespace

unsigned int* device_error_word(int* cuda_err, volatile unsigned int** mirror) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *cuda_err = static_cast<int>(e != cudaSuccess ? e : cudaErrorInvalidDevice);
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_error_mu);
  ErrorHandles& h = g_error_cache[dev];
  const unsigned long long ctx = current_context_id();
  if (h.word == nullptr || h.ctx != ctx) {
    // first use in this context (or the context changed: a device reset
    // ended the old one): look the word up with this device current, which
    // also creates the context if none exists yet
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_error_block);
    if (e != cudaSuccess) {
      *cuda_err = static_cast<int>(e);
      return nullptr;
    }
    h.word = static_cast<unsigned int*>(ptr);
    h.mirror = nullptr;
    // The mirror: best effort; without it the kernels still record errors in
    // the device word, and only the host's early refusal is lost.
    if (!g_mirror_registered && !g_mirror_failed) {
      e = cudaHostRegister(g_mirror_page, sizeof(g_mirror_page),
                           cudaHostRegisterPortable | cudaHostRegisterMapped);
      if (e == cudaSuccess || e == cudaErrorHostMemoryAlreadyRegistered) {
        g_mirror_registered = true;
      } else {
        g_mirror_failed = true;
      }
      cudaGetLastError();   // a failed registration must not linger as the last error
    }
    if (g_mirror_registered) {
      unsigned int* slot = g_mirror_page + 16 * dev;
      void* dslot = nullptr;
      if (cudaHostGetDevicePointer(&dslot, slot, 0) == cudaSuccess && dslot != nullptr) {
        // publish the mirror's device address next to the word (synchronous,
        // once per context)
        if (cudaMemcpy(h.word + 2, &dslot, sizeof(dslot), cudaMemcpyHostToDevice) == cudaSuccess)
          h.mirror = slot;
      }
      cudaGetLastError();
    }
    h.ctx = current_context_id();
  }
  *cuda_err = 0;
  if (mirror != nullptr) *mirror = h.mirror;
  return h.word;
}

int read_and_clear_error(void* stream, unsigned int* value, bool clear) {
  int err = 0;
  volatile unsigned int* mirror = nullptr;
  unsigned int* w = device_error_word(&err, &mirror);
  if (w == nullptr) return err;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return static_cast<int>(e);
  unsigned int v = 0;
  e = cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return static_cast<int>(e);
  if (v != 0 && clear) {
    const unsigned int zero = 0;
    e = cudaMemcpy(w, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return static_cast<int>(e);
  }
  if (mirror != nullptr && clear) *mirror = 0u;
  *value = v;
  return 0;
}

}  // namespace ra
