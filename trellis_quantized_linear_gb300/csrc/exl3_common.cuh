// Device helpers shared by the libexl3 kernels (sm_103a).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/exl3.h"
#include "exl3_bounds.cuh"

namespace exl3 {

// Rounds a shared-memory offset up to 1024 bytes.
__host__ __device__ constexpr int align1024(int v) { return (v + 1023) & ~1023; }

// Calls f(std::integral_constant<int, i>{}) for i = 0 .. N-1 (compile-time indices).
template <typename F, int... Is>
__device__ __forceinline__ void static_for_impl(F &&f, std::integer_sequence<int, Is...>) {
  (f(std::integral_constant<int, Is>{}), ...);
}
template <int N, typename F>
__device__ __forceinline__ void static_for(F &&f) {
  static_for_impl(f, std::make_integer_sequence<int, N>{});
}

// ---------------------------------------------------------------------------
// Trellis decode (storage format in include/exl3.h)
// ---------------------------------------------------------------------------

constexpr uint32_t kLcgMul = 89226354u;
constexpr uint32_t kLcgAdd = 64248484u;
constexpr uint32_t kKeepMask = 0x8FFF8FFFu;
constexpr uint32_t kFlipBits = 0x3B603B60u;
// fp32(1/sqrt(128)) = 2^-3.5
constexpr float kInvSqrt128 = 0.0883883476483184405f;

// Masked LCG word of one 16-bit state: two fp16 halves, each in +-[1/8, 2).
__device__ __forceinline__ uint32_t lcg_word(uint32_t state) {
  const uint32_t u = state * kLcgMul + kLcgAdd;
  uint32_t r;
  // (u & kKeepMask) ^ kFlipBits as one three-input logic op (LUT 0x6A).
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(r) : "r"(u), "r"(kKeepMask), "r"(kFlipBits));
  return r;
}

// Weights of two states packed as half2 {lo: state_a, hi: state_b}.
// Each weight is RNE_fp16(lo16 + hi16); the fp16 add computes the exact sum
// rounded to nearest even, and the sum of two halves in +-[1/8, 2) is never
// subnormal, so one packed add is the format's fp32-sum-then-round.
__device__ __forceinline__ uint32_t decode_pair(uint32_t state_a, uint32_t state_b) {
  uint32_t ua = lcg_word(state_a);
  uint32_t ub = lcg_word(state_b);
  uint32_t lo = __byte_perm(ua, ub, 0x5410);  // {ua.lo, ub.lo}
  uint32_t hi = __byte_perm(ua, ub, 0x7632);  // {ua.hi, ub.hi}
  __half2 s = __hadd2(*reinterpret_cast<__half2 *>(&lo), *reinterpret_cast<__half2 *>(&hi));
  return *reinterpret_cast<uint32_t *>(&s);
}

// Per-thread view of four consecutive tile rows (rows 4q..4q+3 of a 16x16
// tile) for a trellis of width BITS.
//
// A thread owns stream words [4q*BITS, 4q*BITS + 4*BITS) of its tile (the
// own bits of its four rows, which start on word boundaries because a tile
// row holds 16*BITS bits) plus the word just before them (circularly; from
// the neighbouring lane). seq[0] is that prefix word and seq[1 + j] is own
// word j. X[j] = seq[j] << 16 | seq[j+1] is the 32-bit MSB-first view of two
// consecutive words, so any 16-bit window inside them is one shift + mask.
template <int BITS>
struct RowWindows {
  static constexpr int kWords = 4 * BITS;  // own words
  uint32_t X[kWords];

  // own: the 4*BITS own words as 2*BITS little-endian uint32 (word 2a in the
  // low half of own[a]); prev: the uint32 holding the prefix word in its
  // high half.
  __device__ __forceinline__ void build(const uint32_t (&own)[2 * BITS], uint32_t prev) {
    // X[0] = prefix << 16 | word0
    X[0] = __byte_perm(own[0], prev, 0x7610);
#pragma unroll
    for (int j = 1; j < kWords; ++j) {
      if (j & 1) {
        // seq[j] = word j-1 (low half of own[(j-1)/2]), seq[j+1] = word j (high half)
        X[j] = __byte_perm(own[(j - 1) >> 1], own[(j - 1) >> 1], 0x1032);
      } else {
        // seq[j] = word j-1 (high half of own[j/2-1]), seq[j+1] = word j (low half of own[j/2])
        X[j] = __byte_perm(own[j >> 1], own[(j >> 1) - 1], 0x7610);
      }
    }
  }

  // The same state with at most one integer-pipe instruction: the view
  // X << k, k = o mod 8, is a multiply by mk[k] = 2^k on the FMA pipe (mk
  // opaque to the compiler, so the multiply is not turned into a shift).
  // The window then starts at bit 16 or 24 of the view: one shift or one
  // byte permute. Two windows of one X word with the same k share the view.
  template <int R, int C>
  __device__ __forceinline__ uint32_t state_fma(const uint32_t (&mk)[8]) const {
    constexpr int s = R * BITS * 16 + (C + 1) * BITS;  // window start, in seq bits
    constexpr int j = s >> 4;
    constexpr int o = s & 15;
    constexpr int k = o & 7;
    static_assert(R >= 0 && R < 4 && C >= 0 && C < 16, "window index out of range");
    static_assert(o == 0 ? (j >= 1 && j <= kWords) : (j >= 0 && j < kWords), "window outside X");
    if constexpr (o == 0) {
      return X[j - 1] & 0xFFFFu;  // seq[j]
    } else if constexpr (k == 0) {
      return __byte_perm(X[j], 0u, 0x4421);  // o == 8
    } else {
      const uint32_t v = X[j] * mk[k];  // window at bits 31-(o-k) .. 16-(o-k), o - k in {0, 8}
      if constexpr (o == k) {
        return v >> 16;
      } else {
        return __byte_perm(v, 0u, 0x4421);
      }
    }
  }

  // 16-bit state of weight c (0..15) of thread row r (0..3).
  template <int R, int C>
  __device__ __forceinline__ uint32_t state() const {
    constexpr int s = R * BITS * 16 + (C + 1) * BITS;  // window start, in seq bits
    constexpr int j = s >> 4;
    constexpr int o = s & 15;
    static_assert(R >= 0 && R < 4 && C >= 0 && C < 16, "window index out of range");
    static_assert(o == 0 ? (j >= 1 && j <= kWords) : (j >= 0 && j < kWords), "window outside X");
    if constexpr (o == 0) {
      return X[j - 1] & 0xFFFFu;  // seq[j]
    } else if constexpr (o == 8) {
      return __byte_perm(X[j], 0u, 0x4421);  // (X >> 8) & 0xFFFF
    } else {
      return (X[j] >> (16 - o)) & 0xFFFFu;
    }
  }
};

// Packed pair {w(state_a), w(state_b)}: both halves of each masked word are
// summed with one fp16 add (operands selected by half), then the two sums are
// packed. Same arithmetic as decode_pair, fewer integer-pipe instructions.
template <bool kPackFma>
__device__ __forceinline__ uint32_t decode_pair_sel(uint32_t state_a, uint32_t state_b) {
  const uint32_t ua = lcg_word(state_a);
  const uint32_t ub = lcg_word(state_b);
  const __half2 ha = *reinterpret_cast<const __half2 *>(&ua);
  const __half2 hb = *reinterpret_cast<const __half2 *>(&ub);
  __half2 r;
  if constexpr (kPackFma) {
  // (w_a, w_a) * (1, 0) + (w_b, w_b) * (0, 1): exact, no integer-pipe op.
  const __half2 ra = __half2half2(__hadd(__low2half(ha), __high2half(ha)));
  const __half2 rb = __half2half2(__hadd(__low2half(hb), __high2half(hb)));
  const __half2 one_zero = __halves2half2(__float2half_rn(1.f), __float2half_rn(0.f));
  const __half2 zero_one = __halves2half2(__float2half_rn(0.f), __float2half_rn(1.f));
  r = __hfma2(ra, one_zero, __hmul2(rb, zero_one));
  } else {
  r = __halves2half2(__hadd(__low2half(ha), __high2half(ha)), __hadd(__low2half(hb), __high2half(hb)));
  }
  return *reinterpret_cast<const uint32_t *>(&r);
}

// Weight of one state in both halves of a half2: one fp16 add of the masked
// word's halves (operands selected by half). An mma A register holding
// {w, w} against a B register holding {x, 0} contributes exactly w * x, so
// no packing of two weights into one register is needed.
__device__ __forceinline__ uint32_t decode_dup(uint32_t state) {
  const uint32_t u = lcg_word(state);
  const __half2 h = *reinterpret_cast<const __half2 *>(&u);
  const __half2 r = __hadd2(__low2half2(h), __high2half2(h));
  return *reinterpret_cast<const uint32_t *>(&r);
}

// The 16 window states of one tile row for BITS = 4. A and B hold the row's
// own words w0..w3 as two little-endian uint32 (w1 << 16 | w0, w3 << 16 | w2);
// P holds the stream word just before the row in its high half. State c is
// the 16-bit window ending at row bit 4c + 3, earliest bit most significant.
// Per row: two byte permutes and two multiplies build the views that
// straddle a register boundary (p|w0, w1|w2, and their 4-bit shifts); the
// 4-bit shifts of w0|w1 and w2|w3 are rotations of A and B; then every state
// is one instruction.
__device__ __forceinline__ void row4_states(uint32_t A, uint32_t B, uint32_t P, uint32_t m16, uint32_t (&s)[16]) {
  const uint32_t xc0 = __byte_perm(A, P, 0x7610);  // p << 16 | w0
  const uint32_t xc1 = __byte_perm(B, A, 0x7610);  // w1 << 16 | w2
  const uint32_t y0 = xc0 * m16, y1 = xc1 * m16;   // the same, 4 bits further (low nibble unused)
  const uint32_t ya = __funnelshift_l(A, A, 20);   // (w0 << 16 | w1) << 4 (low nibble unused)
  const uint32_t yb = __funnelshift_l(B, B, 20);   // (w2 << 16 | w3) << 4
  s[0] = y0 >> 16;
  s[1] = __byte_perm(xc0, 0u, 0x4421);
  s[2] = __byte_perm(y0, 0u, 0x4421);
  s[3] = A & 0xFFFFu;
  s[4] = ya >> 16;
  s[5] = __byte_perm(A, 0u, 0x4403);
  s[6] = __byte_perm(ya, 0u, 0x4421);
  s[7] = A >> 16;
  s[8] = y1 >> 16;
  s[9] = __byte_perm(xc1, 0u, 0x4421);
  s[10] = __byte_perm(y1, 0u, 0x4421);
  s[11] = B & 0xFFFFu;
  s[12] = yb >> 16;
  s[13] = __byte_perm(B, 0u, 0x4403);
  s[14] = __byte_perm(yb, 0u, 0x4421);
  s[15] = B >> 16;
}

// Loads the 8*BITS own bytes of a thread (address 8-byte aligned for every
// BITS, 16-byte aligned for even BITS) into 2*BITS uint32.
template <int BITS, bool kShared>
__device__ __forceinline__ void load_own_words(const uint8_t *p, uint32_t (&own)[2 * BITS]) {
  if constexpr ((BITS & 1) == 0) {
#pragma unroll
    for (int i = 0; i < BITS / 2; ++i) {
      uint4 v;
      if constexpr (kShared) {
        v = *reinterpret_cast<const uint4 *>(p + 16 * i);
      } else {
        v = __ldg(reinterpret_cast<const uint4 *>(p + 16 * i));
      }
      own[4 * i + 0] = v.x;
      own[4 * i + 1] = v.y;
      own[4 * i + 2] = v.z;
      own[4 * i + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < BITS; ++i) {
      uint2 v;
      if constexpr (kShared) {
        v = *reinterpret_cast<const uint2 *>(p + 8 * i);
      } else {
        v = __ldg(reinterpret_cast<const uint2 *>(p + 8 * i));
      }
      own[2 * i + 0] = v.x;
      own[2 * i + 1] = v.y;
    }
  }
}

// Same, from a 32-bit shared-memory address (explicit ld.shared, for buffers
// whose generic pointer has lost its address space).
template <int BITS>
__device__ __forceinline__ void load_own_words_shared(uint32_t saddr, uint32_t (&own)[2 * BITS]) {
  if constexpr ((BITS & 1) == 0) {
#pragma unroll
    for (int i = 0; i < BITS / 2; ++i)
      asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(own[4 * i]), "=r"(own[4 * i + 1]), "=r"(own[4 * i + 2]), "=r"(own[4 * i + 3])
                   : "r"(saddr + 16 * i));
  } else {
#pragma unroll
    for (int i = 0; i < BITS; ++i)
      asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(own[2 * i]), "=r"(own[2 * i + 1]) : "r"(saddr + 8 * i));
  }
}

__device__ __forceinline__ void st_shared_v2(uint32_t saddr, uint32_t a, uint32_t b) {
  asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(saddr), "r"(a), "r"(b) : "memory");
}

// The prefix word of thread (g, q) is the last own word of thread
// (g, (q+3)&3): circular inside the tile's four row-quads.
template <int BITS>
__device__ __forceinline__ uint32_t prefix_from_neighbour(const uint32_t (&own)[2 * BITS], int lane) {
  int src = (lane & ~3) | ((lane + 3) & 3);
  return __shfl_sync(0xffffffffu, own[2 * BITS - 1], src);
}

// ---------------------------------------------------------------------------
// Status word, bounded waits
// ---------------------------------------------------------------------------

constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// The error word keeps the first error since it was last read.
__device__ __forceinline__ void report_timeout(int *status) {
  if (status) atomicCAS(status, 0, (int)EXL3_ERR_DEVICE_TIMEOUT);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test of the phase with the given parity.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait that lets the thread sleep (up to `hint_ns`) until the phase
// completes, so waiting warps leave their issue slots to working ones.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Waits for phase `parity` of an mbarrier to complete. Gives up after
// limit_ns, records EXL3_ERR_DEVICE_TIMEOUT and returns false.
__device__ __forceinline__ bool mbar_wait_limit(uint32_t bar, uint32_t parity, int *status,
                                                unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  unsigned long long t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if ((it & 15u) == 0 && globaltimer_ns() - t0 > limit_ns) {
      report_timeout(status);
      return false;
    }
  }
}

// Same with the library's limit of kWaitLimitNs (2 s).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int *status) {
  return mbar_wait_limit(bar, parity, status, kWaitLimitNs);
}

// Wait used on the error path: same, but with a short limit and no report.
__device__ __forceinline__ void mbar_wait_short(uint32_t bar, uint32_t parity) {
  unsigned long long t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return;
    if ((it & 255u) == 255u && globaltimer_ns() - t0 > 200000000ull) return;
  }
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 1-D bulk copy global -> shared, completing `bytes` on mbarrier `bar`.
// dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// ---------------------------------------------------------------------------
// Host-side launch helpers
// ---------------------------------------------------------------------------

struct DeviceInfo {
  int num_sms = 0;
  int *status = nullptr;  // device address of the error word
  bool ready = false;
};

}  // namespace exl3
