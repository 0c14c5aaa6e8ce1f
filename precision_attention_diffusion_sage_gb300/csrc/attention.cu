// Fused quantized attention forward for sm_103a (INT8 or MXFP4 Q/K, FP8 V).
//
// Restates the kernel described on "[ROCm] Add aiter_sage_attn attention
// backend for gfx1201 (RDNA4)" ("Changes": INT8 QK^T, FP8 PV, FP32
// accumulation, head dim 128, non-causal) and "new MHA v4 entrypoint ..."
// ("Motivation": conditional softmax rescaling, base-2 exponentials,
// pipelines that keep loads, vector ALUs and matrix units busy at once;
// "Technical Details": MXFP4 E2M1 Q/K), with the output plus float32 LSE and
// split-KV of "[None][feat] Add VisualGen FA4 autotuning ..." (first
// paragraph).
//
// GB300 design, per CTA (NQT query tiles of 128 rows of one (b, h)):
//   warps 0 .. 4*NQT-1 : one softmax warpgroup per query tile; thread r owns
//                        row r (TMEM lane r) of its tile.
//   warp 4*NQT         : TMA producer of Q (once) and the K ring.
//   warp 4*NQT+1       : tcgen05 MMA issuer of query tile 0; allocates/frees
//                        TMEM.
//   warp 4*NQT+2       : TMA producer of the V ring (separate so that a K
//                        load never waits for a V slot to free up).
//   warp 4*NQT+3       : tcgen05 MMA issuer of query tile 1 (two tiles), so
//                        that each tile's MMAs wait only for its own softmax.
// TMEM per tile: S (FP32, one column per key of a step) and O (128 FP32
// columns), plus the E8M0 scale factors for MXFP4.
// INT8: S = Q K^T runs as kind::f16 on the codes held as FP16 (sm_103a has no
// 8-bit integer MMA): products and partial sums are integers below 2^24, so
// the FP32 accumulator holds the INT32 dot product exactly. MXFP4: S runs as
// block-scaled kind::mxf4 with the 32-channel scales applied in the MMA.
// Softmax: t = S * alpha, alpha = s_q s_k softmax_scale log2(e) (INT8) or
// softmax_scale log2(e) (MXFP4); the running row reference m is an integer
// (ceil of the maximum), raised only when a step exceeds it by more than
// kHeadroom; O and l are then rescaled by the exact power of two
// 2^(m_old - m_new). P8 = E4M3(2^(t - m + 8 - kHeadroom)) goes to a
// double-buffered 128-byte-swizzled K-major tile in shared memory and
// O += P8 * V8 runs as kind::f8f6f4 with the V tile token-major (an
// MN-major B operand: channels contiguous). Epilogue: O * s_v / l -> BF16,
// LSE = (m + log2 l - 8 + kHeadroom) ln 2 (l is kept in P8 units).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>

#include "attention.cuh"
#include "sm103_ptx.cuh"

namespace sage {
namespace {

constexpr float kLn2 = 0.693147180559945309f;
// Headroom of the running integer maximum (log2 units). The reference m is
// raised (and O, l rescaled by 2^(m_old - m_new)) only when a tile's ceil(max t)
// exceeds m + kHeadroom; otherwise p8 = 2^(t - m + 8 - kHeadroom) <= 2^8 still
// fits E4M3. Every p8 differs from the final-maximum encoding by an exact power
// of two, so the two agree wherever both are normal E4M3 numbers (codes can
// differ only below 2^(kHeadroom - 13) of the row maximum, where this encoding
// is subnormal). A rescale waits for the tile's previous P V, and the tile's
// next step waits for its slowest warp: with a headroom of 2 binades about one
// 128-row tile step in five had a rescaling warp on Gaussian logits (row
// maxima of later tiles often exceed the first tile's by more than 2), with 4
// about one in five hundred.
constexpr float kHeadroom = 4.0f;

// Operand format of Q and K (V is FP8 E4M3 in both).
template <int FMT>
struct QKFormat;
// INT8 codes held as FP16: a 128-row tile is 32 KB, two 64-channel halves in
// the 128-byte swizzled layout. S by kind::f16, one softmax step per 128 keys.
template <>
struct QKFormat<0> {
  static constexpr int kTileBytes = 32768;
  static constexpr int kSfBytes = 0;
  static constexpr int kStep = 128;  // keys per softmax step
};
// MXFP4: rows of 64 bytes of packed E2M1 (64-byte swizzle), 8 KB per 128 rows,
// plus 512 bytes of E8M0 scales per 128 rows staged for the copy to TMEM. S by
// block-scaled kind::mxf4 MMAs in steps of 64 keys: next to two 128-column O
// accumulators and the scale factors, two 128-column S tiles would not fit in
// the 512 TMEM columns.
template <>
struct QKFormat<1> {
  static constexpr int kTileBytes = 8192;
  static constexpr int kSfBytes = 512;
  static constexpr int kStep = 64;
};
// FP8 E4M3: rows of 128 one-byte codes, one 128-byte swizzled box per 128
// rows (16 KB). S by kind::f8f6f4 (the P V kind), one softmax step per 128
// keys; block scales as for INT8.
template <>
struct QKFormat<2> {
  static constexpr int kTileBytes = 16384;
  static constexpr int kSfBytes = 0;
  static constexpr int kStep = 128;
};

// MXFP4 Q/K as format 1, with V and P in MXFP4 too (P V by kind::mxf4).
template <>
struct QKFormat<4> : QKFormat<1> {};

// MXFP4 Q/K (formats 1 and 4) share the S path: 64-key steps, E8M0 scales.
template <int FMT>
__host__ __device__ constexpr bool is_mx() { return FMT == 1 || FMT == 4; }

template <int FMT, int NQT, int STAGES, bool CTA2 = false>
struct SmemLayout {
  using F = QKFormat<FMT>;
  static constexpr int kPSlots = 2 * (128 / F::kStep);  // P slots per query tile
  static constexpr int kQ = 0;                             // NQT Q tiles
  static constexpr int kK = kQ + NQT * F::kTileBytes;      // STAGES K tiles
  static constexpr int kVTile = FMT == 4 ? 8192 : 16384;  // V 128x128: E2M1 V^T or E4M3 V
  // A CTA pair holds half of each K tile (64 keys) and of each V tile (64
  // channels) in each CTA.
  static constexpr int kKStage = CTA2 ? F::kTileBytes / 2 : F::kTileBytes;
  static constexpr int kVStage = CTA2 ? kVTile / 2 : kVTile;
  static constexpr int kV = kK + STAGES * kKStage;         // STAGES V tiles
  static constexpr int kP = kV + STAGES * kVStage;         // NQT x 2 x 16 KB (P, double buffer;
                                                           // also the O staging of the epilogue)
  static constexpr int kSf = kP + NQT * 2 * 16384;         // (NQT + STAGES) scale blocks
  static constexpr int kSv = kSf + (NQT + STAGES) * F::kSfBytes;  // 128 V channel scales
  // MXFP4 V / P (format 4): E8M0 blocks of the V stages and of the P slots,
  // in the line order of the TMEM copy.
  static constexpr int kVsf = kSv + 512;
  static constexpr int kPsf = kVsf + (FMT == 4 ? STAGES * 512 : 0);
  static constexpr int kBar = kPsf + (FMT == 4 ? NQT * kPSlots * 512 : 0);
  // barriers: q_full, k_full[S], k_empty[S], v_full[S], v_empty[S],
  //           s_full[T], s_free[T], p_full[T][kPSlots], o_done[T][kPSlots], mma_final
  static constexpr int kNumBars = 1 + 4 * STAGES + NQT * (2 + 2 * kPSlots) + 1;
  static constexpr int kMisc = kBar + kNumBars * 8;     // tmem slot, abort flag
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kDynamic = kBytes + 1024;        // + alignment slack
};

// TMEM columns of query tile t: S (kStep FP32 columns) and O (128), and for
// MXFP4 the scale factors (4 columns per 128 rows: Q per tile, K in two slots
// that alternate between K tiles).
template <int FMT, int NQT>
struct TmemLayout {
  static constexpr uint32_t kCols = NQT == 1 ? 256 : 512;
  __host__ __device__ static constexpr uint32_t s(int t) { return !is_mx<FMT>() ? t * 256 : NQT * 128 + t * 64; }
  __host__ __device__ static constexpr uint32_t o(int t) { return !is_mx<FMT>() ? t * 256 + 128 : t * 128; }
  __host__ __device__ static constexpr uint32_t sfq(int t) { return NQT * 192 + t * 4; }
  // K scales: two slots per query tile (each tile's MMA warp copies its own).
  __host__ __device__ static constexpr uint32_t sfk(int t, int slot) {
    return NQT * 196 + (t * 2 + slot) * 4;
  }
  // Format 4: V scales in two slots per query tile (alternating V tiles) and
  // P scales in one block per P slot.
  __host__ __device__ static constexpr uint32_t sfv(int t, int slot) {
    return NQT * 196 + (NQT * 2 + t * 2 + slot) * 4;
  }
  __host__ __device__ static constexpr uint32_t sfp(int t, int slot) {
    return NQT * 196 + (NQT * 4 + t * 4 + slot) * 4;
  }
};
static_assert(TmemLayout<1, 2>::sfk(1, 1) + 4 <= TmemLayout<1, 2>::kCols, "TMEM budget");
static_assert(TmemLayout<1, 1>::sfk(0, 1) + 4 <= TmemLayout<1, 1>::kCols, "TMEM budget");
static_assert(TmemLayout<4, 2>::sfp(1, 3) + 4 <= TmemLayout<4, 2>::kCols, "TMEM budget");
static_assert(TmemLayout<4, 1>::sfp(0, 3) + 4 <= TmemLayout<4, 1>::kCols, "TMEM budget");

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Four E4M3 codes packed in a word, element i in bits 8i+7 .. 8i.
__device__ __forceinline__ uint32_t e4m3x4(float e0, float e1, float e2, float e3) {
  uint32_t r;
  asm("{\n .reg .b16 lo, hi;\n"
      " cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n"
      " cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n"
      " mov.b32 %0, {lo, hi};\n}\n"
      : "=r"(r)
      : "f"(e0), "f"(e1), "f"(e2), "f"(e3));
  return r;
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Maximum of N (64 or 128) values: eight independent 3-input-max chains,
// then a tree.
template <int N>
__device__ __forceinline__ float row_max(const float (&s)[N]) {
  static_assert(N % 16 == 0 && N >= 32, "row length");
  float m[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) m[k] = max3f(s[k], s[k + 8], s[k + 16]);
  constexpr int kTail = 24 + (N - 32) / 16 * 16;  // start of the last 8 values
#pragma unroll
  for (int base = 24; base < kTail; base += 16)
#pragma unroll
    for (int k = 0; k < 8; ++k) m[k] = max3f(m[k], s[base + k], s[base + 8 + k]);
#pragma unroll
  for (int k = 0; k < 8; ++k) m[k] = fmaxf(m[k], s[kTail + k]);
  return max3f(max3f(m[0], m[1], m[2]), max3f(m[3], m[4], m[5]), fmaxf(m[6], m[7]));
}

// Maximum of s[B] .. s[B + 31].
template <int B, int N>
__device__ __forceinline__ float max32(const float (&s)[N]) {
  float m[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) m[k] = max3f(s[B + k], s[B + 8 + k], s[B + 16 + k]);
#pragma unroll
  for (int k = 0; k < 8; ++k) m[k] = fmaxf(m[k], s[B + 24 + k]);
  return max3f(max3f(m[0], m[1], m[2]), max3f(m[3], m[4], m[5]), fmaxf(m[6], m[7]));
}

// Eight E2M1 codes packed in a word, element i in bits 4i+3 .. 4i (round to
// nearest even, saturating at 6).
__device__ __forceinline__ uint32_t e2m1x8(const float (&x)[8]) {
  uint32_t r;
  asm("{\n .reg .b8 b0, b1, b2, b3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
      " mov.b32 %0, {b0, b1, b2, b3};\n}\n"
      : "=r"(r)
      : "f"(x[0]), "f"(x[1]), "f"(x[2]), "f"(x[3]), "f"(x[4]), "f"(x[5]), "f"(x[6]), "f"(x[7]));
  return r;
}

// 2^k for an integer-valued k <= 0 (0 below the normal range).
__device__ __forceinline__ float exp2_neg_int(float k) {
  const int ki = static_cast<int>(k);
  return ki < -126 ? 0.0f : __uint_as_float(static_cast<uint32_t>(ki + 127) << 23);
}

template <bool CL = false>
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort,
                                              int* status, long long limit) {
  if (mbar_wait<CL>(bar, parity, abort, limit)) return true;
  if (!*abort) {
    *abort = 1;
    atomicOr(status, kStatusTimeout);
  }
  return false;
}

// Warp-collective variant: every lane waits, the result is uniform. The
// common case (phase already complete) costs one try_wait: the whole warp
// executes it on the same barrier state, so its result is uniform already.
// CL: cluster-scope acquire (barriers the peer CTA of a pair arrives on or
// completes copies on).
template <bool CL = false>
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          int* status, long long limit) {
  if (CL ? mbar_try_wait_cl(bar, parity) : mbar_try_wait(bar, parity)) return true;
  const bool r = wait_or_abort<CL>(bar, parity, abort, status, limit);
  return __all_sync(0xffffffffu, r);
}

// Bounded wait that ignores the abort flag (used to drain in-flight work,
// which always completes; so it keeps the default bound).
template <bool CL = false>
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, int* status) {
  const int zero = 0;
  if (!mbar_wait<CL>(bar, parity, &zero)) atomicOr(status, kStatusTimeout);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// Dot product of row r of an INT8 Q tile (FP16-held codes, two 64-channel
// halves of 128 rows x 128 B at +0 and +16 KB, 16-byte chunks swizzled by
// r & 7) with 128 channel values in global memory.
__device__ __forceinline__ float q_dot_kmean(uint32_t tile, int r, const float* mu) {
  float acc = 0.0f;
#pragma unroll
  for (int hlf = 0; hlf < 2; ++hlf)
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      const uint32_t addr = tile + hlf * 16384 + r * 128 + (((g ^ r) & 7) << 4);
      uint32_t w[4];
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                   : "r"(addr));
      const float4 m0 = __ldg(reinterpret_cast<const float4*>(mu + hlf * 64 + g * 8));
      const float4 m1 = __ldg(reinterpret_cast<const float4*>(mu + hlf * 64 + g * 8 + 4));
      const float mv[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 c = __half22float2(*reinterpret_cast<const __half2*>(&w[q]));
        acc = fmaf(c.x, mv[2 * q], acc);
        acc = fmaf(c.y, mv[2 * q + 1], acc);
      }
    }
  return acc;
}

// Threads per CTA: 7 warps for one query tile; 12 (three full warpgroups)
// for two, so that registers can be moved to the softmax warpgroups with
// setmaxnreg (each SM sub-partition holds one warp of every warpgroup).
template <int NQT>
constexpr int attn_threads() { return NQT == 1 ? 7 * 32 : 12 * 32; }
template <int FMT, int NQT>
__host__ __device__ constexpr bool attn_split_regs() { return !is_mx<FMT>() && NQT == 2; }

// DS: Q smoothing's dS is added to the logits (INT8 only; a separate
// instance, so the plain path keeps its register allocation).
// CTA2: 2-CTA tiles. The grid's CTAs form clusters of two (CTAs 2c and
// 2c + 1, on an SM pair); the even CTA's MMA warps issue cta_group::2 MMAs of
// M = 256 rows (its tile t and its peer's tile t) for both. Each CTA loads
// its own Q tiles, keys 64r .. 64r + 63 of every K tile and channels 64r ..
// 64r + 63 of every V tile (r = its rank in the pair), so each CTA stages
// half of the K/V bytes of the 1-CTA kernel; the peer's copies complete on
// the even CTA's barriers, and the peer's softmax warps arrive there too.
// Everything else (softmax, epilogue) runs in each CTA on its own rows.
template <int FMT, int NQT, int STAGES, bool DS = false, bool CTA2 = false>
__global__ void __launch_bounds__(attn_threads<NQT>(), 1)
    sage_attn_kernel(const __grid_constant__ CUtensorMap tmQ,
                     const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV,
                     const __grid_constant__ CUtensorMap tmO, const AttnParams p) {
  static_assert(!CTA2 || ((FMT == 0 || FMT == 2) && NQT == 2 && !DS), "2-CTA tiles: INT8/FP8");
  using L = SmemLayout<FMT, NQT, STAGES, CTA2>;
  using F = QKFormat<FMT>;
  using TM = TmemLayout<FMT, NQT>;
  constexpr int kStep = F::kStep;
  constexpr int kSteps = 128 / kStep;      // softmax steps per 128-key tile
  constexpr int kPSlots = L::kPSlots;      // P slots per query tile (2 buffers x kSteps)
  constexpr int kSoftmaxWarps = NQT * 4;
  constexpr int kTmaWarp = kSoftmaxWarps;       // Q and K loads
  constexpr int kMmaWarp = kSoftmaxWarps + 1;   // MMAs of query tile 0; owns TMEM
  constexpr int kMmaWarp1 = kSoftmaxWarps + 3;  // MMAs of query tile 1 (two tiles only)
  constexpr int kTmaVWarp = kSoftmaxWarps + 2;  // V loads
  constexpr bool kSplitRegs = attn_split_regs<FMT, NQT>();

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem + L::kQ;
  uint8_t* sK = smem + L::kK;
  uint8_t* sV = smem + L::kV;
  uint8_t* sP = smem + L::kP;
  uint8_t* sSf = smem + L::kSf;  // MXFP4 scales: NQT query tiles, then STAGES K tiles
  float* sSv = reinterpret_cast<float*>(smem + L::kSv);
  uint8_t* sVsf = smem + L::kVsf;  // format 4: V scale blocks per stage
  uint8_t* sPsf = smem + L::kPsf;  // format 4: P scale blocks per query tile and slot
  constexpr bool kMx = is_mx<FMT>();
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + STAGES;
  uint64_t* v_full = k_empty + STAGES;
  uint64_t* v_empty = v_full + STAGES;
  uint64_t* s_full = v_empty + STAGES;
  uint64_t* s_free = s_full + NQT;
  uint64_t* p_full = s_free + NQT;
  // p_full[t * kPSlots + slot]: all 128 rows of that P slot written. One per
  // slot: a fast warp may finish step u+1 before a slow warp of its
  // warpgroup has arrived for step u, so the two must not share a barrier.
  uint64_t* o_done = p_full + kPSlots * NQT;  // [t * kPSlots + slot]: P V of that slot done
  uint64_t* mma_final = o_done + kPSlots * NQT;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);

  const int warp = static_cast<int>(threadIdx.x >> 5);
  const int lane = static_cast<int>(threadIdx.x & 31);
  // Rank in the CTA pair (0 without pairs); the even CTA issues the MMAs.
  const uint32_t rank = CTA2 ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  // Cluster address of a barrier in the even CTA of the pair.
  auto lead_bar = [&](uint64_t* bar) { return cluster_map(smem_u32(bar), 0); };
  const int64_t h = blockIdx.y;
  const int64_t b = blockIdx.z / p.num_splits;
  const int split = static_cast<int>(blockIdx.z % p.num_splits);
  const int64_t bh = b * p.H + h;
  const int64_t Nq_pad = p.nbq * 128, Nk_pad = p.nbk * 128;

  // A CTA of an earlier launch already ran out of a bounded wait: do not
  // pile further timeouts on top (the status word keeps the error). (Not
  // with pairs: the two CTAs of a pair must take the same path, and the word
  // can change between their reads.)
  if constexpr (!CTA2)
    if (*reinterpret_cast<volatile int*>(p.status) & kStatusTimeout) return;

  // ---- per-batch key range (uniform over the CTA)
  // Token counts fit in 32 bits (the host caps N at 4,194,240).
  int nk = static_cast<int>(p.Nk);
  if (p.k_lens) {
    const int32_t len = p.k_lens[b];
    if (len < 0 || len > p.Nk) {
      if (threadIdx.x == 0) atomicOr(p.status, kStatusDeviceArg);
      return;
    }
    nk = len;
  }
  const int nkv = (nk + 127) / 128;
  const int per_split = (nkv + p.num_splits - 1) / p.num_splits;
  const int j0 = split * per_split;
  const int j1 = j0 + per_split < nkv ? j0 + per_split : nkv;
  const int niter = j1 > j0 ? j1 - j0 : 0;
  // Softmax steps; a last key tile with at most 64 valid keys needs only its
  // first 64-key step.
  int nsteps = niter * kSteps;
  if (kSteps == 2 && niter > 0 && j1 == nkv && nk - (nkv - 1) * 128 <= 64) nsteps -= 1;

  if (niter == 0) {
    // No keys for this (batch, split): empty softmax, O = 0, LSE = -inf.
    if (warp < kSoftmaxWarps) {
      const int t = warp / 4, r = static_cast<int>(threadIdx.x & 127);
      const int64_t row = (static_cast<int64_t>(blockIdx.x) * NQT + t) * 128 + r;
      if (row < p.Nq) {
        if (p.num_splits > 1) {
          float* op = p.o_part + ((static_cast<int64_t>(split) * p.B * p.H + bh) * p.Nq + row) * 128;
          for (int d = 0; d < 128; d += 4) *reinterpret_cast<float4*>(op + d) = make_float4(0, 0, 0, 0);
          p.lse_part[(static_cast<int64_t>(split) * p.B * p.H + bh) * p.Nq + row] = -INFINITY;
        } else {
          __nv_bfloat16* orow = p.o + b * p.osb + row * p.osn + h * p.osh;
          for (int d = 0; d < 128; d += 8) *reinterpret_cast<uint4*>(orow + d) = make_uint4(0, 0, 0, 0);
          if (p.lse) p.lse[bh * p.Nq + row] = -INFINITY;
        }
      }
    }
    return;
  }

  // ---- setup
  // V channel scales (MXFP4 V carries its scales inside the MMA: 1).
  if (threadIdx.x < 128)
    sSv[threadIdx.x] = FMT == 4 ? 1.0f : __ldg(&p.v_scale[bh * 128 + threadIdx.x]);
  // With pairs, the even CTA's barriers that the peer also arrives on count
  // its arrivals: q_full one relay arrive, s_free / p_full one per peer warp
  // (per-warp arrivals in both CTAs: 4 + 4).
  constexpr int kStepArrivals = CTA2 ? 8 : 128;
  if (threadIdx.x == 0) {
    mbar_init(q_full, CTA2 && leader ? 2 : 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], NQT);  // one commit per query tile's MMA warp
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], NQT);
    }
    for (int t = 0; t < NQT; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&s_free[t], kStepArrivals);
      for (int q = 0; q < kPSlots; ++q) {
        mbar_init(&p_full[t * kPSlots + q], kStepArrivals);
        mbar_init(&o_done[t * kPSlots + q], 1);
      }
    }
    mbar_init(mma_final, NQT);
    *abort = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    // One warp of each CTA of a pair allocates, collectively for the pair.
    if constexpr (CTA2) {
      tmem_alloc_pair(tmem_slot, TM::kCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, TM::kCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  // Pairs: both CTAs' barriers are initialised and their TMEM allocated
  // before either CTA signals the other.
  if constexpr (CTA2)
    cluster_sync();
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  // INT8 with two query tiles: 384 threads launch with 168 registers each, a
  // pool of 384 * 168 = 64512 that setmaxnreg redistributes: the two softmax
  // warpgroups take 232 and the producer/MMA warpgroup keeps 40
  // (128 * (232 + 232 + 40) = 64512). The host refuses to launch if the
  // compiled register count would leave the pool smaller than that. (The
  // MXFP4 kernel, with 64-key steps, runs faster without the split.)
  if (warp >= kSoftmaxWarps) {
    if constexpr (kSplitRegs) asm volatile("setmaxnreg.dec.sync.aligned.u32 40;\n" ::: "memory");
  // The producer and MMA warps run their loops warp-converged (every lane
  // waits; values stay warp-uniform, so the TMA coordinates and the MMA
  // descriptors live in uniform registers) and one elected lane issues.
  if (warp == kTmaWarp) {
    // ================================================================ TMA producer (Q, K)
    if constexpr (kMx) {
      // E8M0 scales of the query tiles, written in the order the TMEM copy
      // reads: lane L stores the 16-byte line of rows L, L+32, L+64, L+96.
      for (int t = 0; t < NQT; ++t) {
        const int64_t qt = static_cast<int64_t>(blockIdx.x) * NQT + t;
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        if (qt < p.nbq) {
          const uint32_t* src = p.q_sf + bh * Nq_pad + qt * 128 + lane;
#pragma unroll
          for (int c = 0; c < 4; ++c) w[c] = __ldg(src + 32 * c);
        }
        st_shared_v4(smem_u32(sSf + t * 512) + lane * 16, w[0], w[1], w[2], w[3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
    }
    if (elect_one()) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      mbar_arrive_expect_tx(q_full, NQT * F::kTileBytes);
      for (int t = 0; t < NQT; ++t) {
        const int y = static_cast<int>(bh * Nq_pad + (static_cast<int64_t>(blockIdx.x) * NQT + t) * 128);
        if constexpr (FMT == 0) {
          tma_load_2d(sQ + t * 32768, &tmQ, q_full, 0, y);
          tma_load_2d(sQ + t * 32768 + 16384, &tmQ, q_full, 64, y);
        } else {
          tma_load_2d(sQ + t * F::kTileBytes, &tmQ, q_full, 0, y);
        }
      }
    }
    __syncwarp();
    // MXFP4: the next K tile's scale words, loaded one fill ahead.
    uint32_t kw[4] = {0u, 0u, 0u, 0u};
    const uint32_t* ksf = nullptr;
    if constexpr (kMx) {
      ksf = p.k_sf + bh * Nk_pad + lane;
#pragma unroll
      for (int c = 0; c < 4; ++c) kw[c] = __ldg(ksf + j0 * 128 + 32 * c);
    }
    // Fill `it` goes to stage it % STAGES once the fill STAGES earlier has
    // been consumed; `rph` is the parity of the current round of stages.
    int s = 0, filled = 0;
    uint32_t rph = 0;
    for (int it = 0; it < niter; ++it) {
      if (it >= STAGES && !warp_wait(&k_empty[s], rph ^ 1u, abort, p.status, p.wait_cycles)) break;
      if constexpr (kMx) {
        st_shared_v4(smem_u32(sSf + (NQT + s) * 512) + lane * 16, kw[0], kw[1], kw[2], kw[3]);
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (elect_one()) {
        const int yk = static_cast<int>(bh * Nk_pad) + (j0 + it) * 128;
        if constexpr (CTA2) {
          // This CTA's 64 keys of the tile (64-row boxes), completing on the
          // even CTA's barrier, which expects both halves.
          if (leader) mbar_arrive_expect_tx(&k_full[s], 2 * L::kKStage);
          const uint32_t kb = lead_bar(&k_full[s]);
          const int yh = yk + 64 * static_cast<int>(rank);
          if constexpr (FMT == 0) {
            tma_load_2d_pair(sK + s * L::kKStage, &tmK, kb, 0, yh);
            tma_load_2d_pair(sK + s * L::kKStage + L::kKStage / 2, &tmK, kb, 64, yh);
          } else {
            tma_load_2d_pair(sK + s * L::kKStage, &tmK, kb, 0, yh);
          }
        } else {
          mbar_arrive_expect_tx(&k_full[s], F::kTileBytes);
          if constexpr (FMT == 0) {
            tma_load_2d(sK + s * 32768, &tmK, &k_full[s], 0, yk);
            tma_load_2d(sK + s * 32768 + 16384, &tmK, &k_full[s], 64, yk);
          } else {
            tma_load_2d(sK + s * F::kTileBytes, &tmK, &k_full[s], 0, yk);
          }
        }
      }
      __syncwarp();
      if constexpr (kMx) {
        if (it + 1 < niter) {
#pragma unroll
          for (int c = 0; c < 4; ++c) kw[c] = __ldg(ksf + (j0 + it + 1) * 128 + 32 * c);
        }
      }
      filled = it + 1;
      if (++s == STAGES) {
        s = 0;
        rph ^= 1u;
      }
    }
    // Drain: no TMA write may still be in flight when the CTA exits. (With
    // pairs the even CTA's barriers see both CTAs' K copies complete, and
    // the peer exits only after the final cluster barrier.)
    drain_wait<CTA2>(q_full, 0, p.status);
    if (leader) {
      for (int st = 0; st < STAGES; ++st) {
        const int fills = (filled - st + STAGES - 1) / STAGES;
        if (fills > 0) drain_wait<CTA2>(&k_full[st], static_cast<uint32_t>(fills - 1) & 1u, p.status);
      }
    }
  } else if (warp == kTmaVWarp) {
    // ================================================================ TMA producer (V)
    if (elect_one()) tma_prefetch_desc(&tmV);
    __syncwarp();
    int s = 0, filled = 0;
    uint32_t rph = 0;
    for (int it = 0; it < niter; ++it) {
      // Testing only: no V load at all, so that the P V waits run out (no
      // copy is left in flight: nothing was issued to drain).
      if (p.withhold_v) break;
      if (it >= STAGES && !warp_wait(&v_empty[s], rph ^ 1u, abort, p.status, p.wait_cycles)) break;
      if constexpr (FMT == 4) {
        // The tile's E8M0 scales (128 channel rows x 4 bytes, contiguous),
        // written in the line order of the TMEM copy (line L: rows L, L+32,
        // L+64, L+96), visible to the async proxy before the tile's barrier.
        const uint32_t* vsf = p.v_sf + (bh * p.nbk + j0 + it) * 128 + lane;
        st_shared_v4(smem_u32(sVsf + s * 512) + lane * 16, __ldg(vsf), __ldg(vsf + 32),
                     __ldg(vsf + 64), __ldg(vsf + 96));
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (elect_one()) {
        // E4M3 V: 128 token rows of 128 channel bytes (token-major; with pairs
        // this CTA's 64 channels, completing on the even CTA's barrier).
        // Format 4: E2M1 V^T rows of Nk_pad / 2 bytes.
        const int yv = static_cast<int>(bh * Nk_pad) + (j0 + it) * 128;
        if constexpr (CTA2) {
          if (leader) mbar_arrive_expect_tx(&v_full[s], 2 * L::kVStage);
          tma_load_2d_pair(sV + s * L::kVStage, &tmV, lead_bar(&v_full[s]),
                           64 * static_cast<int>(rank), yv);
        } else if constexpr (FMT == 4) {
          mbar_arrive_expect_tx(&v_full[s], L::kVTile);
          tma_load_2d(sV + s * L::kVTile, &tmV, &v_full[s], (j0 + it) * 64,
                      static_cast<int>(bh * 128));
        } else {
          mbar_arrive_expect_tx(&v_full[s], L::kVTile);
          tma_load_2d(sV + s * L::kVTile, &tmV, &v_full[s], 0, yv);
        }
      }
      __syncwarp();
      filled = it + 1;
      if (++s == STAGES) {
        s = 0;
        rph ^= 1u;
      }
    }
    if (leader) {
      for (int st = 0; st < STAGES; ++st) {
        const int fills = (filled - st + STAGES - 1) / STAGES;
        if (fills > 0) drain_wait<CTA2>(&v_full[st], static_cast<uint32_t>(fills - 1) & 1u, p.status);
      }
    }
  } else if (CTA2 && !leader && warp == kMmaWarp) {
    // ================================================================ pair peer
    // The even CTA issues every MMA; this warp relays the completion of this
    // CTA's Q copies to the even CTA's q_full.
    if (warp_wait(q_full, 0, abort, p.status, p.wait_cycles) && elect_one())
      mbar_arrive_remote(lead_bar(q_full));
    __syncwarp();
  } else if ((!CTA2 || leader) && (warp == kMmaWarp || (NQT == 2 && warp == kMmaWarp1))) {
    // ================================================================ MMA issuers
    // One warp per query tile issues that tile's MMAs, so neither tile's
    // tensor work waits in line behind the other tile's softmax. Both read
    // the same K/V stages; a stage is released once both have committed.
    const int t = warp == kMmaWarp ? 0 : 1;
    // M = 256 rows (this CTA's tile t and the peer's) with pairs.
    constexpr int kM = CTA2 ? 256 : 128;
    constexpr uint32_t kIdescS = idesc_f32acc(kM, 128);  // f16 x f16 -> f32 (INT8 codes)
    constexpr uint32_t kIdescO = idesc_f32acc(kM, 128);  // e4m3 x e4m3 -> f32
    // P V: B = the V tile, token-major in shared memory (channels contiguous):
    // an MN-major operand.
    constexpr uint32_t kIdescPV = idesc_f32acc(kM, 128, true);
    // Descriptor low words of this tile's operand buffers (k slices add a
    // constant). The 64- and 128-byte swizzled layouts share the encoding.
    const uint32_t q_lo = sw128_desc_lo(smem_u32(sQ + t * F::kTileBytes));
    const uint32_t k_lo = sw128_desc_lo(smem_u32(sK));    // + tile bytes / 16 per stage
    const uint32_t p_lo = sw128_desc_lo(smem_u32(sP + t * 2 * 16384));  // + buffer * 1024
    const uint32_t v_lo = sw128_desc_lo(smem_u32(sV));    // + stage * 1024
    const uint32_t d_s = tbase + TM::s(t), d_o = tbase + TM::o(t);
    constexpr int kPSlotShift = kPSlots == 4 ? 2 : 1;  // log2(kPSlots)
    // The elected lane is the same (lowest) lane every time, so the commits
    // track the MMAs that lane issued.
    // S for a step using K stage `stage`, 64-key half `half` (MXFP4) and
    // K-scale TMEM slot `sf_slot`.
    auto issue_s = [&](int stage, int half, int sf_slot) {
      if constexpr (FMT == 0) {
        const uint32_t ka = k_lo + stage * (L::kKStage >> 4);
        if (elect_one()) {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            // K slice k: 64-channel box k / 4 (the Q box is 16 KB, a K box
            // holds the stage's 128, or with pairs 64, keys), 32 bytes each.
            const uint32_t offq = ((k >> 2) * 16384 + (k & 3) * 32) >> 4;
            const uint32_t offk = ((k >> 2) * (L::kKStage / 2) + (k & 3) * 32) >> 4;
            if constexpr (CTA2)
              mma_f16_ss_lo_pair(d_s, q_lo + offq, ka + offk, kIdescS, k > 0);
            else
              mma_f16_ss_lo(d_s, q_lo + offq, ka + offk, kIdescS, k > 0);
          }
          if constexpr (CTA2)
            mma_commit_pair(&s_full[t]);
          else
            mma_commit(&s_full[t]);
        }
      } else if constexpr (FMT == 2) {
        // E4M3 x E4M3 over K = 128: four K = 32 slices of the 128-byte rows.
        const uint32_t ka = k_lo + stage * (L::kKStage >> 4);
        if (elect_one()) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            if constexpr (CTA2)
              mma_f8_ss_lo_pair(d_s, q_lo + k * 2, ka + k * 2, kIdescO, k > 0);
            else
              mma_f8_ss_lo(d_s, q_lo + k * 2, ka + k * 2, kIdescO, k > 0);
          }
          if constexpr (CTA2)
            mma_commit_pair(&s_full[t]);
          else
            mma_commit(&s_full[t]);
        }
      } else {
        // Keys 64h .. 64h+63 of the stage: B rows at +4096 bytes, their
        // scales two TMEM columns further (rows 64..127 of the 128-row copy).
        const uint32_t ka = k_lo + stage * 512 + half * 256;
        const uint32_t sfa = tbase + TM::sfq(t);
        const uint32_t sfb = tbase + TM::sfk(t, sf_slot) + half * 2;
        if (elect_one()) {
          mma_mxf4_ss_lo(d_s, q_lo, ka, idesc_mxf4(128, 64, 0), sfa, sfb, 0u);
          mma_mxf4_ss_lo(d_s, q_lo + 2, ka + 2, idesc_mxf4(128, 64, 2), sfa, sfb, 1u);
          mma_commit(&s_full[t]);
        }
      }
      __syncwarp();
    };
    // MXFP4: scales of K stage `stage` to this tile's TMEM slot `sf_slot`
    // (local K tile index & 1). The slot was last read by this tile's S MMAs
    // of tile i - 2, complete once the S of the step before this tile's
    // first step has been read (its s_free was waited for).
    auto copy_k_scales = [&](int stage, int sf_slot) {
      if (elect_one())
        tmem_cp_sf512(tbase + TM::sfk(t, sf_slot), smem_u32(sSf + (NQT + stage) * 512));
      __syncwarp();
    };
    // P V of one step: P slot `slot`, V stage `stage`, 64-key half `half`;
    // format 4 also V-scale TMEM slot `vslot` (local V tile index & 1).
    auto issue_pv = [&](int slot, int stage, int half, int vslot, bool acc) {
      const int pbuf = slot / kSteps;
      if constexpr (FMT == 4) {
        // E2M1 P (64-byte rows, keys 64h .. 64h+63 at +32 bytes) times E2M1
        // V^T rows, one K = 64 block-scaled MMA with N = 128 channels; the
        // scale bytes of this half are bytes 2h, 2h+1 of each row's word.
        // The copies precede the MMA in this thread's issue order. A V slot
        // is rewritten two V tiles later and a P slot kPSlots steps later,
        // after the S of this tile's current step completed, which completes
        // only after every earlier MMA of this warp (the reads of the slot).
        const uint32_t pa = p_lo + pbuf * 1024 + half * 2;
        const uint32_t va = v_lo + stage * (L::kVTile >> 4) + half * 2;
        const uint32_t sfa = tbase + TM::sfp(t, slot), sfb = tbase + TM::sfv(t, vslot);
        if (elect_one()) {
          if (half == 0) tmem_cp_sf512(sfb, smem_u32(sVsf + stage * 512));
          tmem_cp_sf512(sfa, smem_u32(sPsf + (t * kPSlots + slot) * 512));
          mma_mxf4_ss_lo(d_o, pa, va, idesc_mxf4(128, 128, 2u * half), sfa, sfb, acc ? 1u : 0u);
          mma_commit(&o_done[t * kPSlots + slot]);
        }
      } else {
        // V stage: 128 token rows of 128 channel bytes in the 128-byte
        // swizzled layout (with pairs 64 channel bytes, 64-byte swizzle); the
        // K = 32 slice kk of P's keys is V's rows 32 kk .. 32 kk + 31.
        const uint32_t pa = p_lo + pbuf * 1024, va = v_lo + stage * (L::kVStage >> 4);
        constexpr uint32_t kVSliceStep = (32 * (CTA2 ? 64 : 128)) >> 4;
        constexpr int kK = kStep / 32;  // K = 32 slices per step
        if (elect_one()) {
#pragma unroll
          for (int k = 0; k < kK; ++k) {
            const int kk = half * kK + k;
            if constexpr (CTA2)
              mma_f8_ss_lo_pair<kSw64DescHi>(d_o, pa + kk * 2, va + kk * kVSliceStep, kIdescPV,
                                             (acc || k > 0) ? 1u : 0u);
            else
              mma_f8_ss_lo(d_o, pa + kk * 2, va + kk * kVSliceStep, kIdescPV,
                           (acc || k > 0) ? 1u : 0u);
          }
          if constexpr (CTA2)
            mma_commit_pair(&o_done[t * kPSlots + slot]);
          else
            mma_commit(&o_done[t * kPSlots + slot]);
        }
      }
      __syncwarp();
    };
    // Commits of the ring stages and of the final barrier reach both CTAs of
    // a pair (each CTA's producers and softmax wait on their own barriers).
    auto commit = [&](uint64_t* bar) {
      if (elect_one()) {
        if constexpr (CTA2)
          mma_commit_pair(bar);
        else
          mma_commit(bar);
      }
      __syncwarp();
    };
    // K ring position of the S steps (stage, parity of its fill round) and
    // V ring position of the P V steps; both advance after a tile's last step.
    int ks = 0, vs = 0;
    uint32_t kph = 0, vph = 0;
    bool ok = warp_wait<CTA2>(q_full, 0, abort, p.status, p.wait_cycles);
    if (ok) ok = warp_wait<CTA2>(&k_full[0], 0, abort, p.status, p.wait_cycles);
    tc_fence_after();
    if (ok) {
      if constexpr (kMx) {
        if (elect_one()) tmem_cp_sf512(tbase + TM::sfq(t), smem_u32(sSf + t * 512));
        __syncwarp();
        copy_k_scales(0, 0);
      }
      issue_s(0, 0, 0);
      if constexpr (kSteps == 1) {
        commit(&k_empty[0]);
        if (++ks == STAGES) { ks = 0; kph ^= 1u; }
      }
    }
    for (int u = 0; ok && u < nsteps; ++u) {
      // Next S first (it needs only the softmax warpgroup to have read the
      // previous S), then this step's P V. V is waited for only right before
      // the P V MMAs.
      const int v = u + 1;
      if (v < nsteps) {
        const int hv = v & (kSteps - 1);
        if (hv == 0) {
          if (!(ok = warp_wait<CTA2>(&k_full[ks], kph, abort, p.status, p.wait_cycles))) break;
          tc_fence_after();
        }
        if (!(ok = warp_wait<CTA2>(&s_free[t], static_cast<uint32_t>(u) & 1u, abort, p.status,
                                   p.wait_cycles)))
          break;
        tc_fence_after();
        const int sf_slot = (v / kSteps) & 1;
        if constexpr (kMx) {
          if (hv == 0) copy_k_scales(ks, sf_slot);
        }
        issue_s(ks, hv, sf_slot);
        if (hv == kSteps - 1) {
          commit(&k_empty[ks]);
          if (++ks == STAGES) { ks = 0; kph ^= 1u; }
        }
      }
      const int hu = u & (kSteps - 1);
      const int slot = u & (kPSlots - 1);
      if (hu == 0) {
        if (!(ok = warp_wait<CTA2>(&v_full[vs], vph, abort, p.status, p.wait_cycles))) break;
        tc_fence_after();
      }
      if (!(ok = warp_wait<CTA2>(&p_full[t * kPSlots + slot],
                                 static_cast<uint32_t>(u >> kPSlotShift) & 1u, abort, p.status,
                                 p.wait_cycles)))
        break;
      tc_fence_after();
      issue_pv(slot, vs, hu, (u / kSteps) & 1, u > 0);
      if (hu == kSteps - 1) {
        commit(&v_empty[vs]);
        if (++vs == STAGES) { vs = 0; vph ^= 1u; }
      }
    }
    // All MMAs issued by both MMA warps must finish before TMEM is freed.
    commit(mma_final);
    drain_wait(mma_final, 0, p.status);
  }
  } else {
      if constexpr (kSplitRegs) asm volatile("setmaxnreg.inc.sync.aligned.u32 232;\n" ::: "memory");
    // ================================================================ softmax
    const int t = warp / 4;
    // Step handshakes with the MMA warp: every thread arrives, or with pairs
    // one lane per warp (after the warp's own accesses, ordered before it by
    // __syncwarp) on the even CTA's barrier.
    auto step_arrive = [&](uint64_t* bar) {
      if constexpr (CTA2) {
        __syncwarp();
        if (lane == 0) {
          if (leader)
            mbar_arrive(bar);
          else
            mbar_arrive_remote(lead_bar(bar));
        }
      } else {
        mbar_arrive(bar);
      }
    };
    const int r = static_cast<int>(threadIdx.x & 127);
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tbase + lane_base + TM::s(t);
    const uint32_t tO = tbase + lane_base + TM::o(t);
    const int64_t qt = static_cast<int64_t>(blockIdx.x) * NQT + t;
    const int64_t row = qt * 128 + r;
    // INT8 / FP8: logit multiplier s_q s_k softmax_scale log2(e) per K tile. MXFP4:
    // the block scales are inside S already, the multiplier is constant.
    float alpha_q = p.scale_log2;
    const float* kscale = nullptr;
    float sk_next = 1.0f;  // K block scale, loaded one tile ahead
    float sq = 0.0f;       // Q block scale (INT8 / FP8)
    if constexpr (!kMx) {
      sq = qt < p.nbq ? __ldg(&p.q_scale[bh * p.nbq + qt]) : 0.0f;
      alpha_q = sq * p.scale_log2;
      kscale = p.k_scale + bh * p.nbk;
      sk_next = __ldg(&kscale[j0]);
    }
    float m = -INFINITY;  // running integer row maximum (log2 units)
    float l = 0.0f;       // running row sum of 2^(t - m + 8)
    bool ok = true;
    const uint32_t p_row0 = smem_u32(sP + (t * 2) * 16384) + r * 128;  // P buffer 0; buffer 1 at +16 KB
    const uint32_t swz = static_cast<uint32_t>(r & 7);
    // Format 4: 64-byte P rows (64-byte swizzle: chunk c at c ^ ((r / 2) & 3))
    // and this row's word in the P scale blocks (line r % 32, word r / 32).
    const uint32_t p_row0_4 = smem_u32(sP + (t * 2) * 16384) + r * 64;
    const uint32_t swz64 = static_cast<uint32_t>((r >> 1) & 3);
    const uint32_t psf_row = smem_u32(sPsf + t * kPSlots * 512) + (r & 31) * 16 + (r >> 5) * 4;

    constexpr int kPSlotShift = kPSlots == 4 ? 2 : 1;  // log2(kPSlots)
    float sk = 1.0f;
    for (int u = 0; u < nsteps; ++u) {
      const int iu = u / kSteps;
      const int hu = u & (kSteps - 1);
      const int j = j0 + iu;
      if constexpr (!kMx) {
        sk = sk_next;
        if (iu + 1 < niter) sk_next = __ldg(&kscale[j + 1]);
      }
      if (!(ok = warp_wait(&s_full[t], static_cast<uint32_t>(u) & 1u, abort, p.status, p.wait_cycles))) break;
      tc_fence_after();
      float s[kStep];
      {
        uint32_t v[kStep];
        if constexpr (kStep == 128)
          tmem_ld128(tS, v);
        else
          tmem_ld64(tS, v);
#pragma unroll
        for (int i = 0; i < kStep; ++i) s[i] = __uint_as_float(v[i]);
      }
      tc_fence_before();
      step_arrive(&s_free[t]);

      // Kept strictly positive, so that a masked score (-inf) gives x = -inf
      // and p = 0 with no per-element test in the exponential loop. A zero
      // scale (an all-zero block) only has exact-zero scores, for which
      // FLT_MIN gives the same x as zero would.
      float alpha = fmaxf(alpha_q * sk, 1.17549435e-38f);
      const int key0 = j * 128 + hu * kStep;
      const int nvalid = nk - key0 < kStep ? nk - key0 : kStep;
      if (nvalid < kStep) {  // keys past the end: -inf, p = 0
#pragma unroll
        for (int c = 0; c < kStep; ++c)
          if (c >= nvalid) s[c] = -INFINITY;
      }
      if constexpr (DS) {
        // Q smoothing: every logit of this query block gains dS_j (natural
        // units, the same for all rows), read through L1 (uniform addresses)
        // after a prefetch one key tile ahead. s becomes the natural-unit
        // logit S s_q s_k + dS_j and the multiplier softmax_scale log2(e).
        static_assert(FMT == 0, "dS is defined for the INT8 format");
        if (qt < p.nbq) {
          const float* dsr = p.delta_s + (bh * p.nbq + qt) * Nk_pad + key0;
          if (lane == 0 && iu + 1 < niter)
            asm volatile("prefetch.global.L1 [%0];" ::"l"(dsr + 128 + (warp & 3) * 32));
          const float beta = fmaxf(sq * sk, 1.17549435e-38f);  // > 0: -inf stays -inf
          const float2 beta2 = make_float2(beta, beta);
#pragma unroll
          for (int c = 0; c < kStep; c += 4) {
            const float4 d = __ldg(reinterpret_cast<const float4*>(dsr + c));
            const float2 t01 = __ffma2_rn(make_float2(s[c], s[c + 1]), beta2, make_float2(d.x, d.y));
            const float2 t23 = __ffma2_rn(make_float2(s[c + 2], s[c + 3]), beta2, make_float2(d.z, d.w));
            s[c] = t01.x;
            s[c + 1] = t01.y;
            s[c + 2] = t23.x;
            s[c + 3] = t23.y;
          }
          alpha = p.scale_log2;
        }
      }
      // Format 4 also keeps the maxima of the two 32-key blocks (P's scales).
      float bm0 = 0.0f, bm1 = 0.0f, mx;
      if constexpr (FMT == 4) {
        bm0 = max32<0>(s);
        bm1 = max32<32>(s);
        mx = fmaxf(bm0, bm1);
      } else {
        mx = row_max<kStep>(s);
      }
      const float cand = ceilf(mx * alpha);
      // First step: set the reference. Later: raise it only past the headroom.
      const float m_new = (u == 0) ? cand : (cand > m + kHeadroom ? cand : m);
      const bool rescale = (u > 0) && (m_new > m);
      if (__any_sync(0xffffffffu, rescale)) {
        // Conditional rescale: O_t must hold P V up to the previous step.
        const int ps = (u - 1) & (kPSlots - 1);
        if (!(ok = warp_wait(&o_done[t * kPSlots + ps],
                             static_cast<uint32_t>((u - 1) >> kPSlotShift) & 1u, abort, p.status, p.wait_cycles)))
          break;
        tc_fence_after();
        const float f = rescale ? exp2_neg_int(m - m_new) : 1.0f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld32(tO + c * 32, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * f);
          tmem_st32(tO + c * 32, v);
        }
        tc_fence_before();
        l *= f;
      }
      m = m_new;
      const int slot = u & (kPSlots - 1);
      if constexpr (FMT == 4) {
        // MXFP4 P per 32 keys: x = S alpha - m, exponent e = floor(max x) - 2
        // (clamped to the E8M0 range; an empty block gives -127), codes
        // E2M1(2^(x - e)) into this row of the 64-byte swizzled P slot and the
        // bytes e + 127 into byte 2h, 2h + 1 of the row's scale word. The codes
        // depend on x - floor(max x) only, not on m; l sums the unquantized
        // 2^x. The slot is free as argued for the FP8 P below.
        float e[2] = {floorf(fmaf(bm0, alpha, -m)) - 2.0f, floorf(fmaf(bm1, alpha, -m)) - 2.0f};
        if (!(e[0] >= -127.0f)) e[0] = -127.0f;
        if (!(e[1] >= -127.0f)) e[1] = -127.0f;
        const uint32_t p_row = p_row0_4 + static_cast<uint32_t>(slot / kSteps) * 16384;
        const float2 alpha2 = make_float2(alpha, alpha);
        float lsum = 0.0f;
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
          const float2 bias2 = make_float2(-m - e[blk], -m - e[blk]);
          float2 acc = make_float2(0.0f, 0.0f);
          uint32_t pk[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float ev[8];
#pragma unroll
            for (int i = 0; i < 8; i += 2) {
              const int c = blk * 32 + q * 8 + i;
              const float2 x = __ffma2_rn(make_float2(s[c], s[c + 1]), alpha2, bias2);
              ev[i] = ex2_approx(x.x);
              ev[i + 1] = ex2_approx(x.y);
              acc = __fadd2_rn(acc, make_float2(ev[i], ev[i + 1]));
            }
            pk[q] = e2m1x8(ev);
          }
          lsum += (acc.x + acc.y) * exp2_neg_int(e[blk]);
          const uint32_t chunk = static_cast<uint32_t>(hu * 2 + blk);  // 16-byte chunk of the row
          st_shared_v4(p_row + ((chunk ^ swz64) << 4), pk[0], pk[1], pk[2], pk[3]);
        }
        l += lsum;
        const uint32_t sfw = (static_cast<uint32_t>(e[0] + 127.0f) |
                              (static_cast<uint32_t>(e[1] + 127.0f) << 8)) << (16 * hu);
        asm volatile("st.shared.b32 [%0], %1;" ::"r"(psf_row + slot * 512), "r"(sfw) : "memory");
      } else {
        const float bias = 8.0f - kHeadroom - m;
        const uint32_t p_row = p_row0 + static_cast<uint32_t>(slot / kSteps) * 16384;
        // The P slot was last read by P V of step u - kPSlots. No wait is
        // needed for it: the MMA warp issued that P V before the S of step u
        // (its loop issues S of step w + 1 after P V of step w - 1, and
        // u - kPSlots <= u - 2), and the s_full commit this warp waited for
        // completes only after every earlier MMA of that warp.
        // x = S * alpha + (8 - m) two at a time (packed FP32x2 FMA), p8 = 2^x,
        // four partial row sums (packed FP32x2 adds).
        const float2 alpha2 = make_float2(alpha, alpha), bias2 = make_float2(bias, bias);
        float2 acc0 = make_float2(0.0f, 0.0f), acc1 = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int ch = 0; ch < kStep / 16; ++ch) {
          uint32_t pk[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int c = ch * 16 + q * 4;
            const float2 x01 = __ffma2_rn(make_float2(s[c + 0], s[c + 1]), alpha2, bias2);
            const float2 x23 = __ffma2_rn(make_float2(s[c + 2], s[c + 3]), alpha2, bias2);
            const float2 e01 = make_float2(ex2_approx(x01.x), ex2_approx(x01.y));
            const float2 e23 = make_float2(ex2_approx(x23.x), ex2_approx(x23.y));
            acc0 = __fadd2_rn(acc0, e01);
            acc1 = __fadd2_rn(acc1, e23);
            pk[q] = e4m3x4(e01.x, e01.y, e23.x, e23.y);
          }
          // 16-byte chunk of this step's keys within the 128-key P row.
          const uint32_t chunk = static_cast<uint32_t>(hu * (kStep / 16) + ch);
          st_shared_v4(p_row + ((chunk ^ swz) << 4), pk[0], pk[1], pk[2], pk[3]);
        }
        l += (acc0.x + acc0.y) + (acc1.x + acc1.y);
      }
      fence_proxy_async_smem();
      step_arrive(&p_full[t * kPSlots + slot]);
    }

    // ---- epilogue
    if (ok)
      ok = warp_wait(&o_done[t * kPSlots + ((nsteps - 1) & (kPSlots - 1))],
                     static_cast<uint32_t>((nsteps - 1) >> kPSlotShift) & 1u, abort, p.status, p.wait_cycles);
    if (ok) {
      tc_fence_after();
      const float inv_l = 1.0f / l;
      // K smoothing took the per-row constant softmax_scale * q^ . mean_k out
      // of every logit (O is unchanged by it); the LSE adds it back, in log2
      // units alpha_q * (q8 . mean_k), from this row's codes in the Q tile.
      float lse_add = 0.0f;
      if constexpr (FMT == 0) {
        if (p.k_mean && (ok = warp_wait(q_full, 0, abort, p.status, p.wait_cycles)))
          lse_add = alpha_q * q_dot_kmean(smem_u32(sQ + t * 32768), r, p.k_mean + bh * 128);
      }
      // l is in units of P: 2^(8 - kHeadroom) times 2^(t - m) for the FP8 P,
      // 2^(t - m) for the MXFP4 P.
      constexpr float kLUnits = FMT == 4 ? 0.0f : 8.0f - kHeadroom;
      const float lse = (m + log2f(l) - kLUnits + lse_add) * kLn2;
      const bool store = row < p.Nq;
      if (p.num_splits > 1) {
        float* op = p.o_part + ((static_cast<int64_t>(split) * p.B * p.H + bh) * p.Nq + row) * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld32(tO + c * 32, v);
          if (store) {
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
              float4 o4;
              o4.x = __uint_as_float(v[i + 0]) * (sSv[c * 32 + i + 0] * inv_l);
              o4.y = __uint_as_float(v[i + 1]) * (sSv[c * 32 + i + 1] * inv_l);
              o4.z = __uint_as_float(v[i + 2]) * (sSv[c * 32 + i + 2] * inv_l);
              o4.w = __uint_as_float(v[i + 3]) * (sSv[c * 32 + i + 3] * inv_l);
              *reinterpret_cast<float4*>(op + c * 32 + i) = o4;
            }
          }
        }
        if (store) p.lse_part[(static_cast<int64_t>(split) * p.B * p.H + bh) * p.Nq + row] = lse;
      } else if (p.o_tma) {
        // Row r as BF16 into this tile's two P buffers (free now: the last
        // P V has completed), laid out as the two 64-channel halves of the
        // 128-byte swizzled box the O tensor map stores from; one thread
        // stores every tile after the final barrier.
        const uint32_t obase = smem_u32(sP + t * 2 * 16384) + r * 128;
        const uint32_t rsw = static_cast<uint32_t>(r & 7);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld32(tO + c * 32, v);
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const float4 sa = *reinterpret_cast<const float4*>(sSv + c * 32 + g * 8);
            const float4 sb = *reinterpret_cast<const float4*>(sSv + c * 32 + g * 8 + 4);
            const float sc[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float a0 = __uint_as_float(v[g * 8 + 2 * k]) * (sc[2 * k] * inv_l);
              const float a1 = __uint_as_float(v[g * 8 + 2 * k + 1]) * (sc[2 * k + 1] * inv_l);
              const __nv_bfloat162 h2 = __floats2bfloat162_rn(a0, a1);
              w[k] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            const uint32_t chunk = static_cast<uint32_t>((c & 1) * 4 + g);
            st_shared_v4(obase + (c >> 1) * 16384 + ((chunk ^ rsw) << 4), w[0], w[1], w[2], w[3]);
          }
        }
        fence_proxy_async_smem();
        if (store && p.lse) p.lse[bh * p.Nq + row] = lse;
      } else {
        __nv_bfloat16* orow = p.o + b * p.osb + row * p.osn + h * p.osh;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld32(tO + c * 32, v);
          if (store) {
#pragma unroll
            for (int i = 0; i < 32; i += 8) {
              uint32_t w[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const float a0 = __uint_as_float(v[i + 2 * k]) * (sSv[c * 32 + i + 2 * k] * inv_l);
                const float a1 = __uint_as_float(v[i + 2 * k + 1]) * (sSv[c * 32 + i + 2 * k + 1] * inv_l);
                const __nv_bfloat162 h2 = __floats2bfloat162_rn(a0, a1);
                w[k] = *reinterpret_cast<const uint32_t*>(&h2);
              }
              *reinterpret_cast<uint4*>(orow + c * 32 + i) = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
        if (store && p.lse) p.lse[bh * p.Nq + row] = lse;
      }
    }
  }

  tc_fence_before();
  // Pairs: the even CTA's MMAs (which write this CTA's tensor memory and read
  // its shared memory) are complete and neither CTA signals the other any
  // more once both have reached this barrier.
  if constexpr (CTA2)
    cluster_sync();
  else
    __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    if constexpr (CTA2)
      tmem_dealloc_pair(tbase, TM::kCols);
    else
      tmem_dealloc(tbase, TM::kCols);
  } else if (warp == kTmaWarp && p.o_tma && !*abort) {
    // Store the staged O tiles (rows past Nq are clipped by the tensor map).
    if (elect_one()) {
      for (int t = 0; t < NQT; ++t) {
        const int qt = static_cast<int>(blockIdx.x) * NQT + t;
        if (qt >= p.nbq) break;
        tma_store_4d(&tmO, sP + t * 2 * 16384, 0, static_cast<int>(h), qt * 128, static_cast<int>(b));
        tma_store_4d(&tmO, sP + t * 2 * 16384 + 16384, 64, static_cast<int>(h), qt * 128,
                     static_cast<int>(b));
      }
      tma_store_commit();
      tma_store_wait_read();
    }
    __syncwarp();
  }
}

// Split-KV merge: one warp per output row, 4 channels per lane.
__global__ void __launch_bounds__(256) merge_splits_kernel(const AttnParams p) {
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = static_cast<int>(threadIdx.x & 31);
  const int64_t rows = p.B * p.H * p.Nq;
  if (gw >= rows) return;
  const int64_t bh = gw / p.Nq, row = gw % p.Nq;
  const int64_t b = bh / p.H, h = bh % p.H;
  const int64_t stride = p.B * p.H * p.Nq;
  float mx = -INFINITY;
  for (int s = 0; s < p.num_splits; ++s) mx = fmaxf(mx, p.lse_part[s * stride + gw]);
  float4 acc = make_float4(0, 0, 0, 0);
  float lse = -INFINITY;
  if (mx != -INFINITY) {
    float wsum = 0.0f;
    for (int s = 0; s < p.num_splits; ++s) {
      const float ls = p.lse_part[s * stride + gw];
      const float w = ls == -INFINITY ? 0.0f : expf(ls - mx);
      wsum += w;
      const float4 o = *reinterpret_cast<const float4*>(p.o_part + (s * stride + gw) * 128 + lane * 4);
      acc.x += w * o.x; acc.y += w * o.y; acc.z += w * o.z; acc.w += w * o.w;
    }
    const float inv = 1.0f / wsum;
    acc.x *= inv; acc.y *= inv; acc.z *= inv; acc.w *= inv;
    lse = mx + logf(wsum);
  }
  __nv_bfloat16* orow = p.o + b * p.osb + row * p.osn + h * p.osh + lane * 4;
  const __nv_bfloat162 h0 = __floats2bfloat162_rn(acc.x, acc.y);
  const __nv_bfloat162 h1 = __floats2bfloat162_rn(acc.z, acc.w);
  uint2 w;
  w.x = *reinterpret_cast<const uint32_t*>(&h0);
  w.y = *reinterpret_cast<const uint32_t*>(&h1);
  *reinterpret_cast<uint2*>(orow) = w;
  if (lane == 0 && p.lse) p.lse[bh * p.Nq + row] = lse;
}

// ------------------------------------------------------------------ host side
bool make_map_2d(CUtensorMap* m, const void* ptr, CUtensorMapDataType dt, int esize,
                 uint64_t inner, uint64_t rows, uint32_t box_inner, uint32_t box_rows,
                 CUtensorMapSwizzle swizzle) {
  const uint64_t dims[2] = {inner, rows};
  const uint64_t strides[1] = {inner * static_cast<uint64_t>(esize)};
  const uint32_t box[2] = {box_inner, box_rows};
  return encode_tiled(m, dt, 2, ptr, dims, strides, box, swizzle);
}

template <int FMT, int NQT, int STAGES, bool DS = false, bool CTA2 = false>
cudaError_t launch_variant(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                           const CUtensorMap& mo, const AttnParams& p, cudaStream_t stream) {
  using L = SmemLayout<FMT, NQT, STAGES, CTA2>;
  static_assert(L::kDynamic <= 232448, "shared memory budget");
  constexpr auto kern = sage_attn_kernel<FMT, NQT, STAGES, DS, CTA2>;
  cudaError_t e = once_per_device<kern>([]() {
    cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kDynamic);
    if (r != cudaSuccess) return r;
    if constexpr (attn_split_regs<FMT, NQT>()) {
      // setmaxnreg can only hand out the registers the CTA was launched with.
      cudaFuncAttributes fa;
      if ((r = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess) return r;
      if (static_cast<long>(fa.numRegs) * attn_threads<NQT>() < 128L * (232 + 232 + 40))
        return cudaErrorInvalidConfiguration;
    }
    return cudaSuccess;
  });
  if (e != cudaSuccess) return e;
  const unsigned ctas_x = static_cast<unsigned>((p.nbq + NQT - 1) / NQT);
  dim3 grid(CTA2 ? (ctas_x + 1) / 2 * 2 : ctas_x, static_cast<unsigned>(p.H),
            static_cast<unsigned>(p.B * p.num_splits));
  if constexpr (CTA2) {
    // Clusters of two CTAs along x (an even grid: a last CTA past the query
    // tiles computes rows that are not stored).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(attn_threads<NQT>());
    cfg.dynamicSmemBytes = L::kDynamic;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, mo, p);
  } else {
    kern<<<grid, attn_threads<NQT>(), L::kDynamic, stream>>>(mq, mk, mv, mo, p);
    return cudaGetLastError();
  }
}

}  // namespace

int attn_q_tiles_per_cta(int64_t nbq) { return nbq >= 2 ? 2 : 1; }

bool attn_cta2_supported(int fmt, int64_t Nq, bool delta_s) {
  return (fmt == 0 || fmt == 2) && !delta_s && attn_q_tiles_per_cta(pad128(Nq) / 128) == 2;
}

// The library's choice between 1-CTA and 2-CTA tiles, from measurement on
// GB300 (every configuration timed both ways): 1-CTA tiles everywhere.
bool attn_prefer_cta2(int fmt, int64_t B, int64_t H, int64_t Nq, int64_t Nk) {
  (void)fmt;
  (void)B;
  (void)H;
  (void)Nq;
  (void)Nk;
  return false;
}

int attn_auto_splits(int64_t B, int64_t H, int64_t Nq, int64_t Nk) {
  const int64_t nbq = pad128(Nq) / 128, nkv = pad128(Nk) / 128;
  const int nqt = attn_q_tiles_per_cta(nbq);
  const int64_t ctas = (nbq + nqt - 1) / nqt * B * H;
  if (ctas >= 152 || nkv < 4) return 1;
  int64_t s = (2 * 152 + ctas - 1) / ctas;
  if (s > nkv / 2) s = nkv / 2;
  if (s > 16) s = 16;
  if (s * B > 65535) s = 65535 / B;
  return s < 1 ? 1 : static_cast<int>(s);
}

cudaError_t launch_attention(const AttnLaunch& a, cudaStream_t stream) {
  const int64_t Nq_pad = pad128(a.p.Nq), Nk_pad = pad128(a.p.Nk);
  const uint64_t q_rows = static_cast<uint64_t>(a.p.B * a.p.H * Nq_pad);
  const uint64_t k_rows = static_cast<uint64_t>(a.p.B * a.p.H * Nk_pad);
  CUtensorMap mq, mk, mv;
  bool maps_ok;
  // 2-CTA tiles: each CTA of a pair loads 64 keys of a K tile and 64
  // channels of a V tile (64-row K boxes, 64-byte V boxes).
  const bool cta2 = a.cta2 != 0;
  const uint32_t kv_rows = cta2 ? 64 : 128;
  if (a.fmt == 0)  // FP16-held INT8 codes: 128-byte boxes of 64 channels
    maps_ok = make_map_2d(&mq, a.q, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, 128, q_rows, 64, 128,
                          CU_TENSOR_MAP_SWIZZLE_128B) &&
              make_map_2d(&mk, a.k, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, 128, k_rows, 64, kv_rows,
                          CU_TENSOR_MAP_SWIZZLE_128B);
  else if (a.fmt == 2)  // E4M3 codes: one 128-byte row per token
    maps_ok = make_map_2d(&mq, a.q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 128, q_rows, 128, 128,
                          CU_TENSOR_MAP_SWIZZLE_128B) &&
              make_map_2d(&mk, a.k, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 128, k_rows, 128, kv_rows,
                          CU_TENSOR_MAP_SWIZZLE_128B);
  else  // packed E2M1: one 64-byte row per token
    maps_ok = make_map_2d(&mq, a.q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 64, q_rows, 64, 128,
                          CU_TENSOR_MAP_SWIZZLE_64B) &&
              make_map_2d(&mk, a.k, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 64, k_rows, 64, 128,
                          CU_TENSOR_MAP_SWIZZLE_64B);
  // E4M3 V: token rows of 128 channel bytes, like an FP8 K tile (128-byte
  // boxes; with pairs 64-byte boxes of one CTA's channels, 64-byte swizzle).
  // Format 4: packed E2M1 V^T rows of Nk_pad / 2 bytes (64-byte boxes, the
  // layout of a K tile).
  if (!maps_ok ||
      !(a.fmt == 4 ? make_map_2d(&mv, a.v, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1,
                                 static_cast<uint64_t>(Nk_pad / 2),
                                 static_cast<uint64_t>(a.p.B * a.p.H * 128), 64, 128,
                                 CU_TENSOR_MAP_SWIZZLE_64B)
                   : make_map_2d(&mv, a.v, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 128, k_rows,
                                 cta2 ? 64 : 128, 128,
                                 cta2 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B)))
    return cudaErrorInvalidValue;
  // O through a 4-D map over the caller's [B][Nq][H][D] strides (boxes of
  // 128 rows x 64 channels); the kernel falls back to direct stores when the
  // strides cannot be described (e.g. a zero stride) or the keys are split.
  AttnParams p = a.p;
  CUtensorMap mo;
  p.o_tma = 0;
  if (p.num_splits <= 1) {
    const uint64_t dims[4] = {128, static_cast<uint64_t>(p.H), static_cast<uint64_t>(p.Nq),
                              static_cast<uint64_t>(p.B)};
    const uint64_t strides[3] = {static_cast<uint64_t>(p.osh) * 2, static_cast<uint64_t>(p.osn) * 2,
                                 static_cast<uint64_t>(p.osb) * 2};
    const uint32_t box[4] = {64, 1, 128, 1};
    if (p.osh > 0 && p.osn > 0 && p.osb > 0 &&
        encode_tiled(&mo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, p.o, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B))
      p.o_tma = 1;
  }
  if (!p.o_tma) mo = mv;  // unused by the kernel
  const bool two = attn_q_tiles_per_cta(p.nbq) == 2;
  if (cta2 && (!two || p.delta_s || (a.fmt != 0 && a.fmt != 2))) return cudaErrorInvalidValue;
  cudaError_t e;
  if (a.fmt == 0)
    e = p.delta_s ? (two ? launch_variant<0, 2, 2, true>(mq, mk, mv, mo, p, stream)
                         : launch_variant<0, 1, 3, true>(mq, mk, mv, mo, p, stream))
                  : (cta2  ? launch_variant<0, 2, 4, false, true>(mq, mk, mv, mo, p, stream)
                     : two ? launch_variant<0, 2, 2>(mq, mk, mv, mo, p, stream)
                           : launch_variant<0, 1, 3>(mq, mk, mv, mo, p, stream));
  else if (a.fmt == 2)
    e = cta2  ? launch_variant<2, 2, 4, false, true>(mq, mk, mv, mo, p, stream)
        : two ? launch_variant<2, 2, 4>(mq, mk, mv, mo, p, stream)
              : launch_variant<2, 1, 4>(mq, mk, mv, mo, p, stream);
  else if (a.fmt == 4)
    e = two ? launch_variant<4, 2, 4>(mq, mk, mv, mo, p, stream)
            : launch_variant<4, 1, 4>(mq, mk, mv, mo, p, stream);
  else
    e = two ? launch_variant<1, 2, 4>(mq, mk, mv, mo, p, stream)
            : launch_variant<1, 1, 4>(mq, mk, mv, mo, p, stream);
  if (e != cudaSuccess || a.p.num_splits <= 1) return e;
  const int64_t rows = a.p.B * a.p.H * a.p.Nq;
  const int64_t blocks = (rows * 32 + 255) / 256;
  merge_splits_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(a.p);
  return cudaGetLastError();
}

}  // namespace sage
