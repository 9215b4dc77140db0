// Decode over keys and values spread across c shards on the sm_103a tensor
// cores: split-K partial states per block, merged afterwards
// ("06 - Sequence / Context Parallelism", section 7: attention of a new query
// over distributed keys is a gather of partial results, like a split-K).
//
// A block owns the (at most 16) query rows of one (batch, key/value head) --
// the G heads sharing the head times the new tokens -- and a fixed set of
// 128-key tiles (tile pi, pi + P, ... over all shards' tiles), and writes one
// partial online-softmax state (o, m, l) for them.  The 16 query rows are too
// few for the M of tcgen05.mma, so the products are taken transposed, with the
// 128 keys (or the output columns) as M = 128 and the 16 query rows as N:
//   S^T = K Q^T        A = K tile (K-major), B = Q (K-major)      -> TMEM, lane = key
//   O^T += V^T P^T     A = V tile read M-major, B = P^T (K-major) -> TMEM, lane = column
// (head dimension D = 128 or 64; for D = 64 lanes 64-127 of O^T are unused).
// Each softmax thread owns one key of the tile (one TMEM lane): it scales and
// masks its 16 scores, the block's maximum per query row is reduced across the
// 128 threads (shuffles, then four warps through shared memory), it writes its
// 16 probabilities into the P^T operand as a bf16 head plus a bf16 remainder
// (so P enters the product with about 16 bits, and the result stays within
// 1e-4 of the float64 definition) and keeps its own share of the row sums.
// Heads and remainders are stacked as the operand's 32 rows, so one N = 32
// product per 16 keys accumulates both into separate columns of O^T (an
// instruction costs the tensor core the same for any N up to 128), added in
// the epilogue.  Every thread also owns one output column of O^T.  Two such
// softmax pipelines (warps 0-3 and 4-7) take the block's tiles in turn, each
// with its own S and P buffers, O^T accumulator and online-softmax state, so
// that one works on a tile while the other's product runs; their two states
// are merged at the end of the block.  K and V tiles stream through three
// shared-memory stages by TMA (a striped shard's keys, every c-th row, through a 5-D view of
// the tensor), so the block reads each key and value byte once, and the
// kernel is bound by HBM bandwidth; the loads carry an evict-first L2 policy,
// so that the stream displaces its own lines rather than whatever else L2
// holds (often lines that would first have to be written back).
//
// Warp roles (320 threads): warps 0-3 and 4-7 the two softmax pipelines
// (even and odd tiles), warp 8 TMA loads, warp 9 tensor-memory allocation;
// its lane 0 issues the MMAs.  Every wait is
// bounded (ra_wait.cuh).

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cstdint>
#include <cstring>

#include "ra_internal.h"
#include "ra_wait.cuh"
#include "sm103_ptx.cuh"

namespace ra {
namespace {

constexpr int kDTRows = 16;           // query rows per block: the MMAs' N
constexpr int kDTKeys = 128;          // keys per tile
constexpr int kDTStages = 3;
constexpr int kDTWarpLoad = 8;
constexpr int kDTWarpMma = 9;
constexpr int kDTThreads = 10 * 32;
constexpr uint32_t kDTTmemCols = 128;  // S0 | S1 (16 columns each) | O0 | O1 (heads, remainders: 32 each)
constexpr int kDTTargetBlocks = 152;  // one resident block per SM

// Shared memory of the kernel for head dimension D (64 or 128).
template <int D>
struct DTSmem {
  static constexpr int kBox = 64;                            // bf16 columns per 128-byte row
  static constexpr int kNB = D / kBox;                       // column boxes per key or value row
  static constexpr int kKVBox = kDTKeys * kBox * 2;          // 16 KB: 128 keys x 64 columns
  static constexpr int kKVTile = kNB * kKVBox;               // 128 keys x D columns
  static constexpr int kRowsBox = kDTRows * kBox * 2;        // 2 KB: 16 rows x 64 columns
  static constexpr int kQ = 0;                               // Q: 16 rows x D columns (kNB boxes)
  static constexpr int kPBox = 2 * kRowsBox;                 // 4 KB: 32 rows (16 heads, 16 remainders) x 64 keys
  static constexpr int kPBuf = 2 * kPBox;                    // P^T for the 128 keys of a tile
  static constexpr int kP = kQ + 2 * kRowsBox;               // two such buffers
  static constexpr int kV = kP + 2 * kPBuf;
  static constexpr int kK = kV + kDTStages * kKVTile;
  static constexpr int kBar = kK + kDTStages * kKVTile;
  // O^T += V^T P^T reads V^T as an M = 128 operand: its rows 64-127 are the
  // second column box of the value tile (D = 128), or, for D = 64, whatever
  // lies one offset further -- the same stage's key tile -- which only fills
  // O^T lanes 64-127, never read (a row of the product depends only on its
  // own row of A)
  static constexpr int kVLbo = (D == 128) ? kKVBox : (kK - kV);
  static constexpr int bKVFull = 0;
  static constexpr int bKVEmpty = bKVFull + kDTStages;
  static constexpr int bSFull = bKVEmpty + kDTStages;
  static constexpr int bPFull = bSFull + 2;
  static constexpr int bPVDone = bPFull + 2;                 // P V of tile j done: [j & 1]
  static constexpr int bXch = bPVDone + 2;                   // row-max exchange, 2 parities
  static constexpr int bDrain = bXch + 2;
  static constexpr int kNumBars = bDrain + 1;
  static constexpr int kMisc = kBar + kNumBars * 8;          // tmem slot, abort flag
  static constexpr int kRed = kMisc + 16;                    // [2 pipelines][4 warps][16] floats
  static constexpr int kComb = kRed + 2 * 4 * kDTRows * 4;   // [2 pipelines][m, l][16] floats
  static constexpr int kQpos = kComb + 2 * 2 * kDTRows * 4;  // [16] ints: the rows' positions
  static constexpr int kBytes = kQpos + kDTRows * 4;
  static constexpr int kDynamic = kBytes + 1024;
  static_assert(kK % 1024 == 0 && kV % 1024 == 0 && kP % 1024 == 0, "swizzle atoms are 1024 bytes");
  static_assert(kDynamic <= 232448, "shared memory budget");
  static_assert(D == 64 || D == 128, "head dimension");
  static_assert(kVLbo % 16 == 0 && kVLbo / 16 < 16384, "leading byte offset field");
};

__device__ __forceinline__ long long dt_natural_key(int r, int i, int n, int c, int layout) {
  if (layout == RA_ZIGZAG) {
    const int ch = n / 2;
    return i < ch ? static_cast<long long>(r) * ch + i : static_cast<long long>(2 * c - 1 - r) * ch + (i - ch);
  }
  if (layout == RA_STRIPED) return r + static_cast<long long>(c) * i;
  return static_cast<long long>(r) * n + i;
}

// Byte offset of element (row, col) of a K-major operand with 128-byte rows
// and the 128-byte swizzle (16-byte chunk c of row r sits at chunk c ^ (r % 8)),
// boxes of box_bytes per 64 columns.
__device__ __forceinline__ uint32_t sw128_offset(int row, int col, int box_bytes) {
  const int box = col >> 6;
  const int k = col & 63;
  return static_cast<uint32_t>(box * box_bytes + row * 128 + (((k >> 3) ^ (row & 7)) << 4) + ((k & 7) << 1));
}

// Maximum (or sum) of 16 per-thread values over the 32 lanes of a warp with
// 16 shuffles: after the call, lane L holds the result for row
// ((L>>4)&1)*8 + ((L>>3)&1)*4 + ((L>>2)&1)*2 + ((L>>1)&1) (lanes L and L^1 agree).
template <bool kMax>
__device__ __forceinline__ float warp_reduce16(const float (&v)[16], int lane) {
  float a8[8], a4[4], a2[2];
  const bool h1 = (lane >> 4) & 1, h2 = (lane >> 3) & 1, h3 = (lane >> 2) & 1, h4 = (lane >> 1) & 1;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float mine = h1 ? v[8 + k] : v[k];
    const float other = h1 ? v[k] : v[8 + k];
    const float r = __shfl_xor_sync(0xffffffffu, other, 16);
    a8[k] = kMax ? fmaxf(mine, r) : mine + r;
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float mine = h2 ? a8[4 + k] : a8[k];
    const float other = h2 ? a8[k] : a8[4 + k];
    const float r = __shfl_xor_sync(0xffffffffu, other, 8);
    a4[k] = kMax ? fmaxf(mine, r) : mine + r;
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const float mine = h3 ? a4[2 + k] : a4[k];
    const float other = h3 ? a4[k] : a4[2 + k];
    const float r = __shfl_xor_sync(0xffffffffu, other, 4);
    a2[k] = kMax ? fmaxf(mine, r) : mine + r;
  }
  const float mine = h4 ? a2[1] : a2[0];
  const float other = h4 ? a2[0] : a2[1];
  const float r = __shfl_xor_sync(0xffffffffu, other, 2);
  float a = kMax ? fmaxf(mine, r) : mine + r;
  const float r1 = __shfl_xor_sync(0xffffffffu, a, 1);
  return kMax ? fmaxf(a, r1) : a + r1;
}

__device__ __forceinline__ int reduced_row(int lane) {
  return ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
}

template <int D>
__global__ void __launch_bounds__(kDTThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const DecodeParams p) {
  using L = DTSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = ptx::smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBar + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);
  const Abort ab{abort_flag, p.err};
  float* const red = reinterpret_cast<float*>(smem + L::kRed);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.Hq / p.Hkv;
  const int rows = G * p.R;
  const int row_blocks = (rows + kDTRows - 1) / kDTRows;
  const int bx = blockIdx.x;
  const int rb = bx % row_blocks;
  const int g = (bx / row_blocks) % p.Hkv;
  const int b = bx / (row_blocks * p.Hkv);
  const int pi = blockIdx.y;
  const int row0 = rb * kDTRows;
  const int nrows = min(kDTRows, rows - row0);
  // A shard is one stretch of the natural order (contiguous; striped through
  // the strided view) or two (zig-zag chunks); each stretch is cut into
  // 128-key tiles of its own, so that every tile is one TMA box.
  const int np = (p.layout == RA_ZIGZAG) ? 2 : 1;   // stretches per shard
  const int pl = p.n / np;                          // keys per stretch
  const int tpp = (pl + kDTKeys - 1) / kDTKeys;     // tiles per stretch
  const int tps = np * tpp;                         // tiles per shard
  const int T = p.c * tps;
  const int J = (pi < T) ? (T - 1 - pi) / p.P + 1 : 0;   // tiles of this block
  // tile j of this block: its shard, the shard-local index of its first key,
  // and its number of keys
  auto tile_of = [&](int j, int& shard, int& i0, int& len) {
    const int ti = pi + j * p.P;
    shard = ti / tps;
    const int rem = ti % tps;
    const int lt = rem % tpp;
    i0 = (rem / tpp) * pl + lt * kDTKeys;
    len = min(kDTKeys, pl - lt * kDTKeys);
  };

  // ---- set-up --------------------------------------------------------------
  if (threadIdx.x == 0) {
    for (int s = 0; s < kDTStages; ++s) {
      ptx::mbar_init(bar(L::bKVFull + s), 1);
      ptx::mbar_init(bar(L::bKVEmpty + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(bar(L::bSFull + i), 1);
      ptx::mbar_init(bar(L::bPFull + i), 128);
      ptx::mbar_init(bar(L::bXch + i), 128);
    }
    ptx::mbar_init(bar(L::bPVDone), 1);
    ptx::mbar_init(bar(L::bPVDone + 1), 1);
    ptx::mbar_init(bar(L::bDrain), 1);
    *abort_flag = (*reinterpret_cast<volatile unsigned int*>(p.err) != 0) ? 1 : 0;
    ptx::fence_mbar_init();
  }
  if (warp == kDTWarpLoad && lane == 0) {
    ptx::tma_prefetch_desc(&tm_k);
    ptx::tma_prefetch_desc(&tm_v);
  }
  if (warp == kDTWarpMma) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kDTTmemCols);
    ptx::tmem_relinquish();
  }
  // the rows' query positions (rows past the block's rows: none visible)
  int* const sqpos = reinterpret_cast<int*>(smem + L::kQpos);
  if (threadIdx.x < kDTRows)
    sqpos[threadIdx.x] = (static_cast<int>(threadIdx.x) < nrows) ? p.q_pos[(row0 + threadIdx.x) % p.R] : INT_MIN;
  // Q: 16 rows x D columns, K-major with the 128-byte swizzle; row
  // n = (head within group) * R + token, rows past the block's rows are zero.
  if (warp < 4) {
    constexpr int kCols = D / 8;       // columns per thread: 8 threads per row
    const int t = threadIdx.x;
    const int n = t >> 3;              // row
    const int d0 = (t & 7) * kCols;
    uint4 w[kCols / 8];
#pragma unroll
    for (int i = 0; i < kCols / 8; ++i) w[i] = make_uint4(0, 0, 0, 0);
    if (n < nrows) {
      const int rr = row0 + n;
      const int h = g * G + rr / p.R;
      const int tok = rr % p.R;
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.q) +
                                                        ((static_cast<long long>(b) * p.R + tok) * p.Hq + h) * D + d0);
#pragma unroll
      for (int i = 0; i < kCols / 8; ++i) w[i] = src[i];
    }
#pragma unroll
    for (int i = 0; i < kCols / 8; ++i)
      *reinterpret_cast<uint4*>(smem + L::kQ + sw128_offset(n, d0 + 8 * i, L::kRowsBox)) = w[i];
    ptx::fence_proxy_async_smem();
  }
  ptx::tc_fence_before_sync();
  __syncthreads();
  ptx::tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == kDTWarpLoad) {
    // ===================== TMA loads of the K and V tiles =================
    if (lane == 0) {
      // every K and V byte is read once: its lines go first when L2 needs room
      const uint64_t pol = ptx::l2_policy_evict_first();
      int issued = 0;
      bool ok = !*abort_flag;
      for (int j = 0; j < J && ok; ++j) {
        const int st = j % kDTStages;
        if (j >= kDTStages) ok = wait_bar(bar(L::bKVEmpty + st), ((j / kDTStages) - 1) & 1u, ab, kErrTimeoutEmpty);
        if (!ok) break;
        int shard, i0, len;
        tile_of(j, shard, i0, len);
        ptx::mbar_arrive_expect_tx(bar(L::bKVFull + st), 2 * L::kKVTile);
        if (p.layout == RA_STRIPED) {
          // every c-th key: (column, head, shard, index in shard, batch)
          for (int x = 0; x < L::kNB; ++x) {
            ptx::tma_load_5d_hint(sbase + L::kK + st * L::kKVTile + x * L::kKVBox, &tm_k, bar(L::bKVFull + st),
                                  x * L::kBox, g, shard, i0, b, pol);
            ptx::tma_load_5d_hint(sbase + L::kV + st * L::kKVTile + x * L::kKVBox, &tm_v, bar(L::bKVFull + st),
                                  x * L::kBox, g, shard, i0, b, pol);
          }
        } else {
          const int nat0 = static_cast<int>(dt_natural_key(shard, i0, p.n, p.c, p.layout));
          for (int x = 0; x < L::kNB; ++x) {
            ptx::tma_load_4d_hint(sbase + L::kK + st * L::kKVTile + x * L::kKVBox, &tm_k, bar(L::bKVFull + st),
                                  x * L::kBox, g, nat0, b, pol);
            ptx::tma_load_4d_hint(sbase + L::kV + st * L::kKVTile + x * L::kKVBox, &tm_v, bar(L::bKVFull + st),
                                  x * L::kBox, g, nat0, b, pol);
          }
        }
        ++issued;
      }
      if (*abort_flag) {
        // let the loads still in flight land before the block exits
        for (int s = 0; s < kDTStages; ++s) {
          const int cnt = (issued > s) ? (issued - 1 - s) / kDTStages + 1 : 0;
          if (cnt > 0) wait_bar_drain(bar(L::bKVFull + s), (cnt - 1) & 1u);
        }
      }
    }
    __syncwarp();
  } else if (warp == kDTWarpMma) {
    // ===================== tensor-core issue ============================
    if (lane == 0) {
      constexpr uint32_t idS = ptx::idesc_bf16_f32(128, kDTRows, false, false);
      constexpr uint32_t idPV = ptx::idesc_bf16_f32(128, 2 * kDTRows, false, true);
      const uint64_t dQ = ptx::smem_desc_sw128(sbase + L::kQ, 16, 1024);
      const uint64_t dK = ptx::smem_desc_sw128(sbase + L::kK, 16, 1024);
      const uint64_t dV = ptx::smem_desc_sw128(sbase + L::kV, L::kVLbo, 1024);
      const uint64_t dP = ptx::smem_desc_sw128(sbase + L::kP, 16, 1024);
      bool ok = true;
      bool issued_any = false;
      auto issue_S = [&](int st, int sb) {
        const uint64_t kd = dK + static_cast<uint64_t>((st * L::kKVTile) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t oa = static_cast<uint64_t>(((kk / 4) * L::kKVBox + (kk % 4) * 32) >> 4);
          const uint64_t ob = static_cast<uint64_t>(((kk / 4) * L::kRowsBox + (kk % 4) * 32) >> 4);
          ptx::tc_mma_ss(tmem + sb * kDTRows, kd + oa, dQ + ob, idS, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_PV = [&](int st, int pb) {
        const uint64_t vd = dV + static_cast<uint64_t>((st * L::kKVTile) >> 4);
        const uint64_t pd = dP + static_cast<uint64_t>((pb * L::kPBuf) >> 4);
#pragma unroll
        for (int kk = 0; kk < kDTKeys / 16; ++kk) {
          // N = 32: the heads of P into O's first 16 columns, the remainders
          // into the next 16; tiles of each parity accumulate into their own O
          const uint64_t oa = static_cast<uint64_t>((kk * 16 * 128) >> 4);
          const uint64_t ob = static_cast<uint64_t>(((kk / 4) * L::kPBox + (kk % 4) * 32) >> 4);
          ptx::tc_mma_ss(tmem + 2 * kDTRows + pb * 2 * kDTRows, vd + oa, pd + ob, idPV, 1u);
        }
      };
      for (int j = 0; j < J && ok; ++j) {
        const int st = j % kDTStages;
        ok = wait_bar(bar(L::bKVFull + st), (j / kDTStages) & 1u, ab, kErrTimeoutK);
        if (!ok) break;
        ptx::tc_fence_after_sync();
        issue_S(st, j & 1);
        ptx::tc_commit(bar(L::bSFull + (j & 1)));
        issued_any = true;
        if (j >= 1) {
          ok = wait_bar(bar(L::bPFull + ((j - 1) & 1)), ((j - 1) >> 1) & 1u, ab, kErrTimeoutP);
          if (!ok) break;
          ptx::tc_fence_after_sync();
          issue_PV((j - 1) % kDTStages, (j - 1) & 1);
          ptx::tc_commit(bar(L::bPVDone + ((j - 1) & 1)));
          ptx::tc_commit(bar(L::bKVEmpty + (j - 1) % kDTStages));
        }
      }
      if (ok && J > 0) {
        ok = wait_bar(bar(L::bPFull + ((J - 1) & 1)), ((J - 1) >> 1) & 1u, ab, kErrTimeoutP);
        if (ok) {
          ptx::tc_fence_after_sync();
          issue_PV((J - 1) % kDTStages, (J - 1) & 1);
          ptx::tc_commit(bar(L::bPVDone + ((J - 1) & 1)));
        }
      }
      if (!ok && issued_any) {
        ptx::tc_commit(bar(L::bDrain));
        if (!wait_bar_drain(bar(L::bDrain), 0)) raise_error(p.err, kErrTimeoutDrain);
      }
    }
    __syncwarp();
  } else {
    // ===================== softmax: thread t owns key t of each tile ========
    // Pipeline sb takes tiles sb, sb + 2, ...: its S and P buffers, its O^T
    // accumulator and its barriers are those of index sb.
    const int sb = warp >> 2;
    const int t = threadIdx.x & 127;                  // also the output column of O^T
    const int wq = warp & 3;                          // TMEM lane quadrant
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_base + sb * kDTRows;
    const uint32_t tO = tmem + lane_base + 2 * kDTRows + sb * 2 * kDTRows;
    {
      uint32_t z[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) z[i] = 0u;
      ptx::tmem_st32(tO, z);
      ptx::tmem_wait_st();
    }
    float m_run[kDTRows], lpart[kDTRows];
#pragma unroll
    for (int n = 0; n < kDTRows; ++n) {
      m_run[n] = -INFINITY;
      lpart[n] = 0.f;
    }
    const float sl2 = p.scale_log2;
    int qmin = INT_MAX;
    for (int n = 0; n < nrows; ++n) qmin = min(qmin, sqpos[n]);
    float* const rbuf = red + sb * 4 * kDTRows;
    uint8_t* const pbuf = smem + L::kP + sb * L::kPBuf;
    bool ok = true;
    int k = 0;                                        // tiles this pipeline has taken
    for (int j = sb; j < J && ok; j += 2, ++k) {
      // where this tile's keys sit (worked out while its S is still on the way)
      int shard, i0, len;
      tile_of(j, shard, i0, len);
      const bool kvalid = t < len;   // rows past the stretch belong to another stretch or lie past the tensor
      const long long pos = dt_natural_key(shard, i0 + (kvalid ? t : 0), p.n, p.c, p.layout);
      // the whole tile visible to every row (the common case): no per-key test
      const bool all_vis = (len == kDTKeys) &&
                           (!p.causal || dt_natural_key(shard, i0 + len - 1, p.n, p.c, p.layout) <= qmin);
      ok = __all_sync(0xffffffffu, wait_bar(bar(L::bSFull + sb), k & 1u, ab, kErrTimeoutS));
      if (!ok) break;
      ptx::tc_fence_after_sync();
      uint32_t su[16];
      ptx::tmem_ld16(tS, su);
      float x[kDTRows];
#pragma unroll
      for (int n = 0; n < kDTRows; ++n) {
        const bool vis = all_vis ? (n < nrows) : (kvalid && n < nrows && (!p.causal || pos <= sqpos[n]));
        x[n] = vis ? __uint_as_float(su[n]) * sl2 : -INFINITY;
      }
      // the tile's maximum per query row: 16 shuffles per warp, then 4 warps
      const float wm = warp_reduce16<true>(x, lane);
      if ((lane & 1) == 0) rbuf[wq * kDTRows + reduced_row(lane)] = wm;
      ptx::mbar_arrive(bar(L::bXch + sb));
      ok = __all_sync(0xffffffffu, wait_bar(bar(L::bXch + sb), k & 1u, ab, kErrTimeoutS));
      if (!ok) break;
      float alpha[kDTRows];
      bool any_rescale = false;
#pragma unroll
      for (int n = 0; n < kDTRows; ++n) {
        const float tmax = fmaxf(fmaxf(rbuf[n], rbuf[kDTRows + n]), fmaxf(rbuf[2 * kDTRows + n], rbuf[3 * kDTRows + n]));
        const float m_new = fmaxf(m_run[n], tmax);
        alpha[n] = (m_run[n] == m_new) ? 1.f : ptx::ex2(m_run[n] - m_new);
        any_rescale |= (alpha[n] != 1.f) && (m_run[n] != -INFINITY);
        m_run[n] = m_new;
      }
      // the P buffer and the accumulator were last used by this pipeline's
      // previous tile, whose P V must have run
      if (k >= 1) {
        ok = __all_sync(0xffffffffu, wait_bar(bar(L::bPVDone + sb), (k - 1) & 1u, ab, kErrTimeoutO));
        if (!ok) break;
        ptx::tc_fence_after_sync();
      }
      // probabilities: this thread's column of P^T (bf16 head and remainder)
      // and its share of l
#pragma unroll
      for (int n = 0; n < kDTRows; ++n) {
        const float muse = (m_run[n] == -INFINITY) ? 0.f : m_run[n];
        const float pr = (x[n] == -INFINITY) ? 0.f : ptx::ex2(x[n] - muse);
        lpart[n] = lpart[n] * alpha[n] + pr;
        const __nv_bfloat16 hi = __float2bfloat16_rn(pr);
        *reinterpret_cast<__nv_bfloat16*>(pbuf + sw128_offset(n, t, L::kPBox)) = hi;
        *reinterpret_cast<__nv_bfloat16*>(pbuf + sw128_offset(kDTRows + n, t, L::kPBox)) =
            __float2bfloat16_rn(pr - __bfloat162float(hi));
      }
      // this thread's column of the accumulator, when a row's maximum rose
      if (any_rescale) {
        uint32_t u[16];
        ptx::tmem_ld16(tO, u);
#pragma unroll
        for (int n = 0; n < kDTRows; ++n) u[n] = __float_as_uint(__uint_as_float(u[n]) * alpha[n]);
        ptx::tmem_st16(tO, u);
        ptx::tmem_ld16(tO + kDTRows, u);
#pragma unroll
        for (int n = 0; n < kDTRows; ++n) u[n] = __float_as_uint(__uint_as_float(u[n]) * alpha[n]);
        ptx::tmem_st16(tO + kDTRows, u);
        ptx::tmem_wait_st();
      }
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before_sync();
      ptx::mbar_arrive(bar(L::bPFull + sb));
    }

    // ---- epilogue: the block's partial state ------------------------------
    // this pipeline's last P V (and with it every product issued before it)
    if (ok && k > 0) {
      ok = __all_sync(0xffffffffu, wait_bar(bar(L::bPVDone + sb), (k - 1) & 1u, ab, kErrTimeoutO));
      if (ok) ptx::tc_fence_after_sync();
    }
    float* const comb = reinterpret_cast<float*>(smem + L::kComb);
    if (ok) {
      // this pipeline's row sums over its 128 threads
      const float ws = warp_reduce16<false>(lpart, lane);
      if ((lane & 1) == 0) rbuf[wq * kDTRows + reduced_row(lane)] = ws;
      ptx::mbar_arrive(bar(L::bXch + sb));
      ok = __all_sync(0xffffffffu, wait_bar(bar(L::bXch + sb), k & 1u, ab, kErrTimeoutS));
      if (ok && t < kDTRows) {
        float mr = -INFINITY;
#pragma unroll
        for (int n = 0; n < kDTRows; ++n)
          if (n == t) mr = m_run[n];
        comb[(sb * 2 + 0) * kDTRows + t] = mr;
        comb[(sb * 2 + 1) * kDTRows + t] =
            rbuf[t] + rbuf[kDTRows + t] + rbuf[2 * kDTRows + t] + rbuf[3 * kDTRows + t];
      }
    }
    // the two pipelines' states meet here (a pipeline that gave up still
    // arrives, so the other never waits in vain)
    ptx::tc_fence_before_sync();
    ptx::named_bar_sync(1, 256);
    ptx::tc_fence_after_sync();
    if (sb == 0 && ok && !*abort_flag) {
      // o = o0 * 2^(m0 - M) + o1 * 2^(m1 - M), l likewise, M = max(m0, m1)
      float f0[kDTRows], f1[kDTRows];
#pragma unroll
      for (int n = 0; n < kDTRows; ++n) {
        const float m0 = comb[n], m1 = comb[2 * kDTRows + n];
        const float M = fmaxf(m0, m1);
        f0[n] = (m0 == -INFINITY) ? 0.f : ptx::ex2(m0 - M);
        f1[n] = (m1 == -INFINITY) ? 0.f : ptx::ex2(m1 - M);
      }
      const uint32_t tO1 = tO + 2 * kDTRows;
      float acc[kDTRows];
      uint32_t u[16];
      ptx::tmem_ld16(tO, u);
#pragma unroll
      for (int n = 0; n < kDTRows; ++n) acc[n] = __uint_as_float(u[n]) * f0[n];
      ptx::tmem_ld16(tO + kDTRows, u);
#pragma unroll
      for (int n = 0; n < kDTRows; ++n) acc[n] = fmaf(__uint_as_float(u[n]), f0[n], acc[n]);
      ptx::tmem_ld16(tO1, u);
#pragma unroll
      for (int n = 0; n < kDTRows; ++n) acc[n] = fmaf(__uint_as_float(u[n]), f1[n], acc[n]);
      ptx::tmem_ld16(tO1 + kDTRows, u);
#pragma unroll
      for (int n = 0; n < kDTRows; ++n) acc[n] = fmaf(__uint_as_float(u[n]), f1[n], acc[n]);
#pragma unroll
      for (int n = 0; n < kDTRows; ++n) {
        if (n >= nrows) break;
        const int rr = row0 + n;
        const int h = g * G + rr / p.R;
        const int tok = rr % p.R;
        // partial layout: o [P, B, R, Hq, D]; m, l [P, B, Hq, R]
        if (t < D) p.part_o[(((static_cast<long long>(pi) * p.B + b) * p.R + tok) * p.Hq + h) * D + t] = acc[n];
      }
      if (t < nrows) {
        const float m0 = comb[t], m1 = comb[2 * kDTRows + t];
        const float M = fmaxf(m0, m1);
        const float l = ((m0 == -INFINITY) ? 0.f : comb[kDTRows + t] * ptx::ex2(m0 - M)) +
                        ((m1 == -INFINITY) ? 0.f : comb[3 * kDTRows + t] * ptx::ex2(m1 - M));
        const int rr = row0 + t;
        const int h = g * G + rr / p.R;
        const int tok = rr % p.R;
        const long long pm = ((static_cast<long long>(pi) * p.B + b) * p.Hq + h) * p.R + tok;
        p.part_m[pm] = M;
        p.part_l[pm] = l;
      }
    }
  }

  // ---- teardown -------------------------------------------------------------
  ptx::tc_fence_before_sync();
  __syncthreads();
  // The merge (a programmatic dependent) may launch once every block has got
  // here: its blocks then land on SMs that are free, spread over the GPU,
  // rather than crowding the few SMs free at the start (where their loads of
  // the partials ran slowly), and the launch itself still overlaps the last
  // blocks' teardown.  The merge waits for this grid's completion before it
  // reads.
  asm volatile("griddepcontrol.launch_dependents;");
  if (warp == kDTWarpMma) {
    ptx::tc_fence_after_sync();
    ptx::tmem_dealloc(tmem, kDTTmemCols);
  }
}

}  // namespace

bool decode_tc_applies(int D, int n, int layout) {
  (void)layout;
  return (D == 64 || D == 128) && n > 0;
}

int decode_tc_partials(int B, int Hkv, int G, int R, int n, int c, int layout) {
  const int np = (layout == RA_ZIGZAG) ? 2 : 1;
  const long long tiles = static_cast<long long>(c) * np * ((n / np + kDTKeys - 1) / kDTKeys);
  const long long units = static_cast<long long>(B) * Hkv * ((static_cast<long long>(G) * R + kDTRows - 1) / kDTRows);
  long long want = (kDTTargetBlocks + units - 1) / units;
  if (want < 1) want = 1;
  if (want > tiles) want = tiles;
  const long long per = (tiles + want - 1) / want;
  return static_cast<int>((tiles + per - 1) / per);
}

template <int D>
int launch_decode_tc_d(const DecodeParams& p, cudaStream_t s) {
  CUtensorMap mk, mv;
  std::memset(&mk, 0, sizeof(mk));
  std::memset(&mv, 0, sizeof(mv));
  launch_stage() = "cuTensorMapEncodeTiled (decode)";
  int e = 0;
  if (p.layout == RA_STRIPED) {
    e = make_tma_map_bf16_strided(&mk, p.k, p.B, p.S, p.Hkv, D, p.c, kDTKeys);
    if (!e) e = make_tma_map_bf16_strided(&mv, p.v, p.B, p.S, p.Hkv, D, p.c, kDTKeys);
  } else {
    e = make_tma_map_bf16(&mk, p.k, p.B, p.S, p.Hkv, D, kDTKeys);
    if (!e) e = make_tma_map_bf16(&mv, p.v, p.B, p.S, p.Hkv, D, kDTKeys);
  }
  if (e) return e;
  // the shared-memory opt-in, once per device (setting it twice is harmless)
  static std::atomic<int> done[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return static_cast<int>(cudaErrorInvalidDevice);
  if (!done[dev].load(std::memory_order_acquire)) {
    launch_stage() = "cudaFuncSetAttribute (decode tensor-core kernel)";
    const cudaError_t ce = cudaFuncSetAttribute(decode_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                DTSmem<D>::kDynamic);
    if (ce != cudaSuccess) return static_cast<int>(ce);
    done[dev].store(1, std::memory_order_release);
  }
  const int G = p.Hq / p.Hkv;
  const int row_blocks = (G * p.R + kDTRows - 1) / kDTRows;
  dim3 grid(static_cast<unsigned>(p.B * p.Hkv * row_blocks), static_cast<unsigned>(p.P));
  launch_stage() = "decode tensor-core kernel launch";
  decode_tc_kernel<D><<<grid, kDTThreads, DTSmem<D>::kDynamic, s>>>(mk, mv, p);
  return static_cast<int>(cudaGetLastError());
}

int launch_decode_tc(const DecodeParams& p, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p.D == 128) return launch_decode_tc_d<128>(p, s);
  if (p.D == 64) return launch_decode_tc_d<64>(p, s);
  return static_cast<int>(cudaErrorInvalidValue);
}

}  // namespace ra
