// Decode over keys and values spread across c shards: split-K partials and
// their merge ("06 - Sequence / Context Parallelism", section 7: with one new
// query the attention over distributed keys needs a gather of partial
// results, like a FlashDecoding split-K).
//
// Every shard's keys are cut into pieces of kPiece local rows.  A thread
// block owns all query rows of one (batch, key/value head) -- the G query
// heads that share the head times the R new tokens, up to 16 rows -- and a
// fixed set of pieces (piece pi, pi + P, pi + 2P, ...), and writes one
// partial online-softmax state (o, m, l) for them; a second kernel merges the
// P partials of every query row in a fixed order.  Each key and value byte is
// read from memory once, so the path is bound by memory bandwidth.
//
// The contraction runs on the tensor cores with warp-level mma.sync
// (m16n8k16, bf16 in, fp32 accumulate): the 16 query rows are exactly the
// instruction's M, which is below the smallest M of tcgen05.mma, and the
// kernel is limited by HBM, not by arithmetic.  Each warp streams 16-key
// chunks of K and V into its own three shared-memory slots with cp.async
// (two chunks in flight while it computes on the third), computes S = Q K^T, keeps a running max and sum per row, and
// accumulates P V with P split into a bf16 head and a bf16 remainder, so the
// probabilities enter the product with about 16 bits of precision (the
// result stays within 1e-4 of the float64 definition).  The four warps'
// states are combined through shared memory in warp order.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <cstring>

#include "ra_internal.h"

namespace ra {
namespace {

constexpr int kDecWarps = 4;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kDecRows = 16;     // query rows (G heads x R tokens) per block: the MMA's M
constexpr int kSub = 16;         // keys per warp step: the MMA's K for P V
constexpr int kPiece = 128;      // shard-local keys per piece
constexpr int kTargetBlocks = 304;   // two resident blocks on each of 152 SMs
constexpr int kStages = 3;           // staged 16-key chunks per warp (two loads in flight)
constexpr int kMergeWarps = 16;   // 56 registers x 512 threads: fits beside a partial block
constexpr int kMergeUnroll = 10;    // partial loads in flight per lane
constexpr int kMergeThreads = kMergeWarps * 32;

template <int D>
struct DecSmem {
  static constexpr int kRow = D + 8;                  // bf16 per staged row (16 bytes of padding)
  static constexpr int kStage = 2 * kSub * kRow;      // K rows then V rows, bf16 elements
  static constexpr int kWarpElems = kStages * kStage;
  static constexpr int kBytes = kDecWarps * kWarpElems * 2;
  static_assert(kDecWarps * kDecRows * D * 4 + 2 * kDecWarps * kDecRows * 4 <= kBytes,
                "the combine buffers reuse the staging area");
};

__device__ __forceinline__ long long natural_key(int r, int i, int n, int c, int layout) {
  if (layout == RA_ZIGZAG) {
    const int ch = n / 2;
    return i < ch ? static_cast<long long>(r) * ch + i : static_cast<long long>(2 * c - 1 - r) * ch + (i - ch);
  }
  if (layout == RA_STRIPED) return r + static_cast<long long>(c) * i;
  return static_cast<long long>(r) * n + i;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global -> shared copy; src_bytes = 0 writes zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

// D (16x8, fp32) += A (16x16, bf16, row) * B (16x8, bf16, col).
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ float fast_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D>
__global__ void __launch_bounds__(kDecThreads)
    decode_partial_kernel(const DecodeParams p) {
  using L = DecSmem<D>;
  constexpr int KS = D / 16;       // k-steps of Q K^T
  constexpr int DT = D / 8;        // 8-column tiles of O
  constexpr int CH = D / 8;        // 16-byte chunks per row
  extern __shared__ __align__(16) uint8_t dsm[];
  __nv_bfloat16* const stage_base = reinterpret_cast<__nv_bfloat16*>(dsm);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int gid = lane >> 2;       // row (and key) index inside an 8-group
  const int tig = lane & 3;
  const int G = p.Hq / p.Hkv;
  const int rows = G * p.R;
  const int row_blocks = (rows + kDecRows - 1) / kDecRows;
  const int bx = blockIdx.x;
  const int rb = bx % row_blocks;
  const int g = (bx / row_blocks) % p.Hkv;
  const int b = bx / (row_blocks * p.Hkv);
  const int pi = blockIdx.y;
  const int row0 = rb * kDecRows;
  const int nrows = min(kDecRows, rows - row0);
  const int pieces = p.c * p.pieces_per_shard;

  // query rows: row = (head within group) * R + token
  int qpos[2];
  bool rvalid[2];
  uint32_t qa[KS][4];
  {
    const __nv_bfloat16* qb = static_cast<const __nv_bfloat16*>(p.q);
    const __nv_bfloat16* qrow[2];
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int r = gid + 8 * hf;
      rvalid[hf] = r < nrows;
      const int rr = row0 + (rvalid[hf] ? r : 0);
      const int h = g * G + rr / p.R;
      const int tok = rr % p.R;
      qpos[hf] = rvalid[hf] ? p.q_pos[tok] : INT_MIN;
      qrow[hf] = qb + ((static_cast<long long>(b) * p.R + tok) * p.Hq + h) * D;
    }
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int hf = i & 1;
        const int col = ks * 16 + 2 * tig + (i >> 1) * 8;
        qa[ks][i] = rvalid[hf] ? *reinterpret_cast<const uint32_t*>(qrow[hf] + col) : 0u;
      }
    }
  }

  asm volatile("griddepcontrol.launch_dependents;");   // the merge may be scheduled early
  float o[DT][4];
#pragma unroll
  for (int i = 0; i < DT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};

  // this warp's work items: (piece, sub-chunk) with pieces pi, pi + P, ...
  // and sub-chunks warp, warp + 4, ... of each piece
  const int subs_per_piece = kPiece / kSub;
  auto item_valid = [&](int pp) { return pp < pieces; };
  __nv_bfloat16* const wbase = stage_base + warp * L::kWarpElems;
  const __nv_bfloat16* kg = static_cast<const __nv_bfloat16*>(p.k);
  const __nv_bfloat16* vg = static_cast<const __nv_bfloat16*>(p.v);

  // Stage the K and V rows of (piece pp, sub-chunk sc) into slot st.
  // Natural position of shard-local key i0 + r for r in [0, 16): affine in r
  // unless the 16 keys straddle the two chunks of a zig-zag shard.
  const int half_n = p.n / 2;
  auto chunk_base = [&](int shard, int i0, long long& nat0, int& step, bool& affine) {
    affine = p.layout != RA_ZIGZAG || ((i0 < half_n) == (i0 + kSub - 1 < half_n));
    step = p.layout == RA_STRIPED ? p.c : 1;
    nat0 = natural_key(shard, i0, p.n, p.c, p.layout);
  };
  const long long row_elems = static_cast<long long>(p.Hkv) * D;     // between key rows
  const __nv_bfloat16* kbg = kg + (static_cast<long long>(b) * p.S * p.Hkv + g) * D;
  const __nv_bfloat16* vbg = vg + (static_cast<long long>(b) * p.S * p.Hkv + g) * D;
  auto issue = [&](int pp, int sc, int st) {
    const int shard = pp / p.pieces_per_shard;
    const int i0 = (pp % p.pieces_per_shard) * kPiece + sc * kSub;
    const int iend = min(p.n, (pp % p.pieces_per_shard + 1) * kPiece);
    long long nat0;
    int step;
    bool affine;
    chunk_base(shard, i0, nat0, step, affine);
    const long long nat_safe = natural_key(shard, 0, p.n, p.c, p.layout);   // rows past the end read nothing
    __nv_bfloat16* ks_ = wbase + st * L::kStage;
    __nv_bfloat16* vs_ = ks_ + kSub * L::kRow;
#pragma unroll
    for (int u = 0; u < kSub * CH / 32; ++u) {
      const int c = lane + 32 * u;
      const int rr = c / CH, cc = c % CH;
      const int i = i0 + rr;
      const bool ok = i < iend;
      long long nat = nat0 + static_cast<long long>(rr) * step;
      if (!affine) nat = natural_key(shard, i, p.n, p.c, p.layout);
      if (!ok) nat = nat_safe;
      const long long off = nat * row_elems + cc * 8;
      cp_async16(smem_u32(ks_ + rr * L::kRow + cc * 8), kbg + off, ok ? 16u : 0u);
      cp_async16(smem_u32(vs_ + rr * L::kRow + cc * 8), vbg + off, ok ? 16u : 0u);
    }
    cp_async_commit();
  };

  auto advance = [&](int& pp_, int& sc_) {
    sc_ += kDecWarps;
    if (sc_ >= subs_per_piece) {
      sc_ = warp;
      pp_ += p.P;
    }
  };
  // the current item and the two after it
  int pp = pi, sc = warp;
  int pp1 = pp, sc1 = sc;
  advance(pp1, sc1);
  int pp2 = pp1, sc2 = sc1;
  advance(pp2, sc2);
  bool have = item_valid(pp), have1 = item_valid(pp1);
  int st = 0;
  if (have) issue(pp, sc, 0);
  if (have1) issue(pp1, sc1, 1);
  while (have) {
    const bool have2 = item_valid(pp2);
    if (have2) issue(pp2, sc2, (st + 2) % kStages);
    // wait for the current chunk; the later ones may stay in flight
    if (have2) cp_async_wait<2>();
    else if (have1) cp_async_wait<1>();
    else cp_async_wait<0>();
    __syncwarp();

    const __nv_bfloat16* ks_ = wbase + st * L::kStage;
    const __nv_bfloat16* vs_ = ks_ + kSub * L::kRow;
    const int shard = pp / p.pieces_per_shard;
    const int pend = min(p.n, (pp % p.pieces_per_shard + 1) * kPiece);
    const int i0 = (pp % p.pieces_per_shard) * kPiece + sc * kSub;

    // ---- S = Q K^T for 16 rows x 16 keys (two 8-key tiles); even and odd
    // k-steps accumulate separately to shorten the dependency chains
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    float s2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    const int krow = (lane >> 4) * 8 + (lane & 7);
    const int kcol = ((lane >> 3) & 1) * 8;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint32_t b00, b01, b10, b11;
      ldsm_x4(smem_u32(ks_ + krow * L::kRow + ks * 16 + kcol), b00, b01, b10, b11);
      if (ks & 1) {
        mma16816(s2[0], qa[ks], b00, b01);
        mma16816(s2[1], qa[ks], b10, b11);
      } else {
        mma16816(s[0], qa[ks], b00, b01);
        mma16816(s[1], qa[ks], b10, b11);
      }
    }
    // ---- mask, running max, probabilities; this lane's four keys
    bool kvis[2][2][2];   // [n-tile][key of the pair][row half]
    long long nat0;
    int step;
    bool affine;
    chunk_base(shard, i0, nat0, step, affine);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        const int r = nt * 8 + 2 * tig + kk;
        const int i = i0 + r;
        const bool in = i < pend;
        const long long pos = affine ? nat0 + static_cast<long long>(r) * step
                                     : natural_key(shard, i, p.n, p.c, p.layout);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) kvis[nt][kk][hf] = in && rvalid[hf] && (!p.causal || pos <= qpos[hf]);
      }
    }
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int hf = e >> 1;
        const float v = s[nt][e] + s2[nt][e];
        s[nt][e] = kvis[nt][e & 1][hf] ? v * p.scale_log2 : -INFINITY;
        mx[hf] = fmaxf(mx[hf], s[nt][e]);
      }
    }
    float alpha[2], muse[2];
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      mx[hf] = fmaxf(mx[hf], __shfl_xor_sync(0xffffffffu, mx[hf], 1));
      mx[hf] = fmaxf(mx[hf], __shfl_xor_sync(0xffffffffu, mx[hf], 2));
      const float m_new = fmaxf(m_run[hf], mx[hf]);
      muse[hf] = (m_new == -INFINITY) ? 0.f : m_new;
      alpha[hf] = (m_run[hf] == m_new) ? 1.f : fast_ex2(m_run[hf] - m_new);
      m_run[hf] = m_new;
    }
    float pr[2][4];
    float psum[2] = {0.f, 0.f};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int hf = e >> 1;
        pr[nt][e] = (s[nt][e] == -INFINITY) ? 0.f : fast_ex2(s[nt][e] - muse[hf]);
        psum[hf] += pr[nt][e];
      }
    }
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) l_run[hf] = l_run[hf] * alpha[hf] + psum[hf];
    if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
      for (int i = 0; i < DT; ++i) {
        o[i][0] *= alpha[0];
        o[i][1] *= alpha[0];
        o[i][2] *= alpha[1];
        o[i][3] *= alpha[1];
      }
    }
    // P as the A operand (k = the 16 keys): a bf16 head and a bf16 remainder
    uint32_t ah[4], al[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int nt = i >> 1, e = (i & 1) * 2;
      const __nv_bfloat162 hv = __floats2bfloat162_rn(pr[nt][e], pr[nt][e + 1]);
      ah[i] = *reinterpret_cast<const uint32_t*>(&hv);
      al[i] = pack_bf16(pr[nt][e] - __low2float(hv), pr[nt][e + 1] - __high2float(hv));
    }
    // ---- O += P V, two 8-column tiles per ldmatrix; the head products for
    // all tiles first, then the remainders, so no two neighbouring MMAs share
    // an accumulator
    const int vrow = ((lane >> 3) & 1) * 8 + (lane & 7);
    const int vcol = (lane >> 4) * 8;
    uint32_t vf[DT / 2][4];
#pragma unroll
    for (int dt = 0; dt < DT; dt += 2)
      ldsm_x4_t(smem_u32(vs_ + vrow * L::kRow + dt * 8 + vcol), vf[dt / 2][0], vf[dt / 2][1], vf[dt / 2][2],
                vf[dt / 2][3]);
#pragma unroll
    for (int dt = 0; dt < DT; dt += 2) {
      mma16816(o[dt], ah, vf[dt / 2][0], vf[dt / 2][1]);
      mma16816(o[dt + 1], ah, vf[dt / 2][2], vf[dt / 2][3]);
    }
#pragma unroll
    for (int dt = 0; dt < DT; dt += 2) {
      mma16816(o[dt], al, vf[dt / 2][0], vf[dt / 2][1]);
      mma16816(o[dt + 1], al, vf[dt / 2][2], vf[dt / 2][3]);
    }
    __syncwarp();
    pp = pp1;
    sc = sc1;
    have = have1;
    pp1 = pp2;
    sc1 = sc2;
    have1 = have2;
    advance(pp2, sc2);
    st = (st + 1) % kStages;
  }

  // ---- the row sums over the four lanes that share a row
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    l_run[hf] += __shfl_xor_sync(0xffffffffu, l_run[hf], 1);
    l_run[hf] += __shfl_xor_sync(0xffffffffu, l_run[hf], 2);
  }
  // ---- combine the four warps' states in warp order
  __syncthreads();   // every warp is done with its staging slots
  float* const ow = reinterpret_cast<float*>(dsm);                       // [warp][row][D]
  float* const wm = ow + kDecWarps * kDecRows * D;                        // [warp][row]
  float* const wl = wm + kDecWarps * kDecRows;
  if (tig == 0) {
    wm[warp * kDecRows + gid] = m_run[0];
    wm[warp * kDecRows + gid + 8] = m_run[1];
    wl[warp * kDecRows + gid] = l_run[0];
    wl[warp * kDecRows + gid + 8] = l_run[1];
  }
  __syncthreads();
  float f[2];
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    const int r = gid + 8 * hf;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, wm[w * kDecRows + r]);
    f[hf] = (m_run[hf] == -INFINITY) ? 0.f : fast_ex2(m_run[hf] - M);
  }
#pragma unroll
  for (int dt = 0; dt < DT; ++dt) {
    float* base = ow + (warp * kDecRows) * D + dt * 8 + 2 * tig;
    *reinterpret_cast<float2*>(base + gid * D) = make_float2(o[dt][0] * f[0], o[dt][1] * f[0]);
    *reinterpret_cast<float2*>(base + (gid + 8) * D) = make_float2(o[dt][2] * f[1], o[dt][3] * f[1]);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < nrows * D; e += kDecThreads) {
    const int r = e / D, d = e % D;
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) acc += ow[(w * kDecRows + r) * D + d];
    const int rr = row0 + r;
    const int h = g * G + rr / p.R;
    const int tok = rr % p.R;
    // partial layout: o [P, B, R, Hq, D]; m, l [P, B, Hq, R]
    p.part_o[(((static_cast<long long>(pi) * p.B + b) * p.R + tok) * p.Hq + h) * D + d] = acc;
    if (d == 0) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, wm[w * kDecRows + r]);
      float Lsum = 0.f;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) {
        const float mw = wm[w * kDecRows + r];
        Lsum += (mw == -INFINITY) ? 0.f : wl[w * kDecRows + r] * fast_ex2(mw - M);
      }
      const long long pm = ((static_cast<long long>(pi) * p.B + b) * p.Hq + h) * p.R + tok;
      p.part_m[pm] = M;
      p.part_l[pm] = Lsum;
    }
  }
}

// One block of 16 warps per (b, h, token) and 32-column slice of the head
// dimension: merge the P partials, normalise, write out (and, from the first
// slice, lse).  Lane = column; the warps take every 16th partial (ten loads
// in flight) and fold them in one online pass; the warps' states are then
// combined, each warp's weight computed by one lane.  Launched as a dependent
// of the partial kernel: the block is small enough to become resident beside
// a partial block, and waits for that grid to finish before it reads the
// partials.
template <int D>
__global__ void __maxnreg__(56) decode_merge_kernel(const DecodeParams p) {
  __shared__ float red_m[kMergeWarps];
  __shared__ float red_l[kMergeWarps];
  __shared__ float red_o[kMergeWarps][32];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const long long row = blockIdx.x;
  const int col = blockIdx.y * 32 + lane;
  const int tok = static_cast<int>(row % p.R);
  const int h = static_cast<int>((row / p.R) % p.Hq);
  const int b = static_cast<int>(row / (static_cast<long long>(p.R) * p.Hq));
  const long long mstride = static_cast<long long>(p.B) * p.Hq * p.R;       // between partials in m, l
  const long long ostride = static_cast<long long>(p.B) * p.R * p.Hq * D;   // between partials in o
  const float* pm = p.part_m + (static_cast<long long>(b) * p.Hq + h) * p.R + tok;
  const float* pl = p.part_l + (static_cast<long long>(b) * p.Hq + h) * p.R + tok;
  const float* po = p.part_o + ((static_cast<long long>(b) * p.R + tok) * p.Hq + h) * D + col;
  float M = -INFINITY, L = 0.f, acc = 0.f;
  static_assert(kMergeUnroll <= 16, "m and l of a round are fetched by lanes 0-15 and 16-31");
  for (int i = warp; i < p.P; i += kMergeUnroll * kMergeWarps) {
    // lane u (< 16) fetches m of the round's partial u, lane 16 + u its l
    const int u_ld = lane & 15;
    const long long i_ld = i + static_cast<long long>(u_ld) * kMergeWarps;
    float ml = (lane < 16) ? -INFINITY : 0.f;
    if (u_ld < kMergeUnroll && i_ld < p.P) ml = (lane < 16) ? pm[i_ld * mstride] : pl[i_ld * mstride];
    float o[kMergeUnroll];
#pragma unroll
    for (int u = 0; u < kMergeUnroll; ++u) {
      const long long ii = i + u * kMergeWarps;
      o[u] = (ii < p.P) ? po[ii * ostride] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kMergeUnroll; ++u) {
      const float mu = __shfl_sync(0xffffffffu, ml, u);
      const float lu = __shfl_sync(0xffffffffu, ml, 16 + u);
      if (mu == -INFINITY) continue;   // an empty partial adds nothing
      const float Mn = fmaxf(M, mu);
      const float a = (M == Mn) ? 1.f : exp2f(M - Mn);
      const float w = (mu == Mn) ? 1.f : exp2f(mu - Mn);
      L = fmaf(lu, w, L * a);
      acc = fmaf(o[u], w, acc * a);
      M = Mn;
    }
  }
  if (lane == 0) {
    red_m[warp] = M;
    red_l[warp] = L;
  }
  red_o[warp][lane] = acc;
  __syncthreads();
  if (warp == 0) {
    // lane w < kMergeWarps holds warp w's state: the block maximum by
    // shuffles, warp w's weight f, and l summed over the warps
    const float mw = (lane < kMergeWarps) ? red_m[lane] : -INFINITY;
    float Mt = mw;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Mt = fmaxf(Mt, __shfl_xor_sync(0xffffffffu, Mt, o));
    const float f = (mw == -INFINITY) ? 0.f : exp2f(mw - Mt);
    float Lt = (lane < kMergeWarps) ? red_l[lane] * f : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Lt += __shfl_xor_sync(0xffffffffu, Lt, o);
    float ot = 0.f;
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) ot = fmaf(red_o[w][lane], __shfl_sync(0xffffffffu, f, w), ot);
    const float inv = (Lt > 0.f) ? 1.f / Lt : 0.f;
    const long long od = ((static_cast<long long>(b) * p.R + tok) * p.Hq + h) * D + col;
    if (p.out_f32)
      static_cast<float*>(p.out)[od] = ot * inv;
    else
      static_cast<__nv_bfloat16*>(p.out)[od] = __float2bfloat16_rn(ot * inv);
    if (lane == 0 && blockIdx.y == 0 && p.lse != nullptr)
      p.lse[(static_cast<long long>(b) * p.Hq + h) * p.R + tok] =
          (Lt > 0.f) ? (Mt + log2f(Lt)) * 0.69314718055994531f : -INFINITY;
  }
}

}  // namespace

int decode_pieces_per_shard(int n) { return (n + kPiece - 1) / kPiece; }

int decode_partials(int B, int Hkv, int G, int R, int pieces) {
  const long long units = static_cast<long long>(B) * Hkv * ((static_cast<long long>(G) * R + kDecRows - 1) / kDecRows);
  long long want = (kTargetBlocks + units - 1) / units;   // blocks per (batch, head, row block)
  if (want < 1) want = 1;
  if (want > pieces) want = pieces;
  const long long per = (pieces + want - 1) / want;        // pieces per block
  return static_cast<int>((pieces + per - 1) / per);
}

template <int D>
int launch_partial(const DecodeParams& p, dim3 grid, cudaStream_t s) {
  // opt in to more than 48 KB of dynamic shared memory (current device)
  static int done[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return static_cast<int>(cudaErrorInvalidDevice);
  if (!done[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(decode_partial_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               DecSmem<D>::kBytes);
    if (e != cudaSuccess) return static_cast<int>(e);
    done[dev] = 1;
  }
  decode_partial_kernel<D><<<grid, kDecThreads, DecSmem<D>::kBytes, s>>>(p);
  return static_cast<int>(cudaGetLastError());
}

int launch_decode(const DecodeParams& p, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int e = 0;
  if (decode_tc_applies(p.D, p.n, p.layout)) {
    e = launch_decode_tc(p, stream);
  } else {
    const int G = p.Hq / p.Hkv;
    const int row_blocks = (G * p.R + kDecRows - 1) / kDecRows;
    dim3 grid(static_cast<unsigned>(p.B * p.Hkv * row_blocks), static_cast<unsigned>(p.P));
    launch_stage() = "decode partial kernel launch";
    e = (p.D == 128) ? launch_partial<128>(p, grid, s) : launch_partial<64>(p, grid, s);
  }
  if (e != 0) return e;
  // The merge may be scheduled while the partial kernel drains; it waits for
  // that grid's completion (programmatic dependent launch) before reading.
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(static_cast<unsigned>(static_cast<long long>(p.B) * p.Hq * p.R),
                     static_cast<unsigned>(p.D / 32));
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr;
  std::memset(&attr, 0, sizeof(attr));
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  launch_stage() = "decode merge kernel launch";
  const cudaError_t me = (p.D == 128) ? cudaLaunchKernelEx(&cfg, decode_merge_kernel<128>, p)
                                      : cudaLaunchKernelEx(&cfg, decode_merge_kernel<64>, p);
  if (me != cudaSuccess) return static_cast<int>(me);
  return static_cast<int>(cudaGetLastError());
}

}  // namespace ra
