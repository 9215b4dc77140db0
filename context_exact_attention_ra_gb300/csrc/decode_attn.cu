// Decode over keys and values spread across c shards: the merge of the
// split-K partials and the launch of both kernels ("06 - Sequence / Context
// Parallelism", section 7: with one new query the attention over distributed
// keys needs a gather of partial results, like a FlashDecoding split-K).
//
// The partial kernel (decode_tc_sm103.cu) writes one online-softmax state
// (o, m, l) per block; the merge below combines the P partials of every query
// row in a fixed order, normalises and writes out and lse.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "ra_internal.h"

namespace ra {
namespace {

constexpr int kMergeWarps = 8;    // 56 registers x 256 threads: fits beside a partial block
constexpr int kMergeUnroll = 19;  // partials per warp and round: 152 partials in one round of loads
constexpr int kMergeThreads = kMergeWarps * 32;

// One block of 8 warps per (b, h, token) and 32-column slice of the head
// dimension: merge the P partials, normalise, write out (and, from the first
// slice, lse).  Lane = column; the warps take every 8th partial, 19 loads in
// flight per lane (up to 152 partials in one round of loads), and fold them:
// the round's maximum by shuffles, each partial's weight on one lane, the
// weighted sums; the warps' states are then combined, each warp's weight
// computed by one lane.  Launched as a programmatic dependent of the partial
// kernel, whose blocks allow the launch as they finish: the block (256
// threads, 56 registers) is small enough to become resident beside a partial
// block still tearing down, and waits for that grid to finish before it reads
// the partials.
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
  static_assert(kMergeUnroll <= 32, "m and l of a round's partial u are fetched by lane u");
  for (int i = warp; i < p.P; i += kMergeUnroll * kMergeWarps) {
    // a round: partials i + u * kMergeWarps, u < kMergeUnroll; lane u fetches
    // that partial's m and l, every lane its column of each partial's o
    const long long i_ld = i + static_cast<long long>(lane) * kMergeWarps;
    const bool has = lane < kMergeUnroll && i_ld < p.P;
    const float mv = has ? pm[i_ld * mstride] : -INFINITY;
    const float lv = has ? pl[i_ld * mstride] : 0.f;
    float o[kMergeUnroll];
#pragma unroll
    for (int u = 0; u < kMergeUnroll; ++u) {
      const long long ii = i + u * kMergeWarps;
      o[u] = (ii < p.P) ? po[ii * ostride] : 0.f;
    }
    // the round's maximum, each partial's weight (one lane each), the
    // weighted sums of l and of the column, folded into the warp's state
    float Mr = mv;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) Mr = fmaxf(Mr, __shfl_xor_sync(0xffffffffu, Mr, off));
    if (Mr == -INFINITY) continue;   // only empty partials (an empty partial adds nothing)
    const float Mn = fmaxf(M, Mr);
    const float wl = (mv == -INFINITY) ? 0.f : exp2f(mv - Mn);
    float lsum = lv * wl;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
    float accr = 0.f;
#pragma unroll
    for (int u = 0; u < kMergeUnroll; ++u) accr = fmaf(o[u], __shfl_sync(0xffffffffu, wl, u), accr);
    const float a = (M == -INFINITY) ? 0.f : exp2f(M - Mn);
    L = fmaf(L, a, lsum);
    acc = fmaf(acc, a, accr);
    M = Mn;
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

int launch_decode(const DecodeParams& p, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!decode_tc_applies(p.D, p.n, p.layout)) return static_cast<int>(cudaErrorInvalidValue);
  const int e = launch_decode_tc(p, stream);
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
