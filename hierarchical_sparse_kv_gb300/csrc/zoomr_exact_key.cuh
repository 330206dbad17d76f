// Exact ranking keys of the ZoomR summary score, and the top-k that ranks them.
//
// The score of segment i for query head h is the inner product alpha = q_h . s_i of the stored bf16 or
// fp32 values (ZoomR page, 3.3 "Per-Head Importance Scoring and Voting", the alpha_i = q^T kbar_i
// equation). The key used here is its exact real value. It is computed with integers, so neither rounding
// nor the order of the additions enters the decision, and a unit's dot products can be split across lanes
// and summed in any order.
//
//   frame    Per unit and side (the group's queries; the unit's summary keys), E is the exponent of the
//            largest magnitude. A value with no bits below 2^(E-55) is an integer multiple of 2^(E-55)
//            below 2^56 in those units, split into two signed 28-bit limbs: hi (multiples of 2^(E-27))
//            and lo (the rest), both with the value's sign.
//   sum      q . s = 2^(Eq+Es-110) * (HH 2^56 + (HL + LH) 2^28 + LL), where HH = sum qh sh, HL = sum qh sl,
//            LH = sum ql sh and LL = sum ql sl are int64 dot products of limbs (|limb| < 2^28 and d <= 128
//            terms keep every partial sum below 2^63), combined into one int128. Only HH is needed when no
//            value has a lower limb, which holds unless a value lies more than about 2^20 below its side's
//            largest. Every hi limb comes from one exact power-of-two multiply and a float-to-int
//            truncation. A pass over the magnitudes marks narrow units (every value within about 2^20 of
//            its side's largest: only HH); elsewhere an exponent test marks the few values that may have
//            a lower limb, and only the warps holding one add the other three products.
//   general  A unit with a value below 2^(E-55) on either side takes a slower path: every product of the
//            integer significands is added at its absolute bit offset into a 640-bit two's-complement
//            accumulator (twenty 32-bit digits), which holds any sum of d <= 128 products of finite bf16
//            or fp32 values exactly.
//
// Ranking is by exact integer comparison, ties to the lower segment index (the spec's tie rule for the
// argtop-k equation of ZoomR 3.3): counting for small n (one thread per segment counts the segments that
// beat it), and a most-significant-digit radix select for larger n.

#pragma once

#include <cuda_bf16.h>

#include <cstddef>
#include <cstdint>

namespace zr {
namespace xk {

constexpr unsigned kAll = 0xFFFFFFFFu;
constexpr int kSlice = 16;      // elements of a row per thread
constexpr int kLimbBits = 28;   // bits per limb
constexpr int kBigDigits = 20;  // 32-bit digits of a general-path key (640 bits)
constexpr int kRadixMinN = 128; // above this many segments the top-k is a radix select

// Bits of the unit flags word (shared memory), OR-ed by the threads that see them.
enum : int { kFlagTail = 1, kFlagDeep = 2, kFlagNonFinite = 4 };

template <typename T>
struct Fmt;
template <>
struct Fmt<__nv_bfloat16> {
  static constexpr int kBits = 16, kMant = 7, kMinLe = -133;
  static constexpr uint32_t kMag = 0x7FFFu, kInf = 0x7F80u;
};
template <>
struct Fmt<float> {
  static constexpr int kBits = 32, kMant = 23, kMinLe = -149;
  static constexpr uint32_t kMag = 0x7FFFFFFFu, kInf = 0x7F800000u;
};

// x = (-1)^neg * M * 2^le for the raw bits u of a finite value (M = 0 for a zero).
template <typename T>
__device__ __forceinline__ void unpack(uint32_t u, uint32_t& M, int& le, bool& neg) {
  using F = Fmt<T>;
  const uint32_t ef = (u >> F::kMant) & 0xFFu, mf = u & ((1u << F::kMant) - 1u);
  M = ef ? (mf | (1u << F::kMant)) : mf;
  le = (ef ? static_cast<int>(ef) : 1) - 127 - F::kMant;
  neg = ((u >> (F::kBits - 1)) & 1u) != 0u;
}

// Exponent of the leading bit of a nonzero finite magnitude.
template <typename T>
__device__ __forceinline__ int top_exp(uint32_t mag) {
  uint32_t M;
  int le;
  bool neg;
  unpack<T>(mag, M, le, neg);
  return le + 31 - __clz(static_cast<int>(M));
}

// Raw bits of element e of a 16-byte vector (e is a compile-time constant after unrolling).
template <typename T>
__device__ __forceinline__ uint32_t elem_bits(const uint4& v, int e) {
  if constexpr (sizeof(T) == 2) {
    const int wi = e >> 1;
    const uint32_t w = wi == 0 ? v.x : wi == 1 ? v.y : wi == 2 ? v.z : v.w;
    return (e & 1) ? (w >> 16) : (w & 0xFFFFu);
  } else {
    return e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
  }
}

template <typename T>
__device__ __forceinline__ uint32_t raw_at(const T* p, int i) {
  if constexpr (sizeof(T) == 2)
    return static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(p)[i]);
  else
    return reinterpret_cast<const uint32_t*>(p)[i];
}

// A non-finite value (unsupported) is ranked as zero and reported through `flags`.
template <typename T>
__device__ __forceinline__ uint32_t finite_or_zero(uint32_t u, int& flags) {
  if ((u & Fmt<T>::kMag) >= Fmt<T>::kInf) {
    flags |= kFlagNonFinite;
    return 0u;
  }
  return u;
}

// The value u in units of 2^(E-55) as two limbs: x = (hi 2^28 + lo) 2^(E-55), both limbs with x's sign.
// Requires |x| < 2^(E+1). Bits of x below 2^(E-55) set kFlagDeep (the limbs then hold x truncated); a
// nonzero lower limb sets kFlagTail.
template <typename T>
__device__ __forceinline__ void to_limbs(uint32_t u, int E, int& hi, int& lo, int& flags) {
  uint32_t M;
  int le;
  bool neg;
  unpack<T>(u, M, le, neg);
  const int sh = le - (E - 55);
  uint32_t vh, vl;
  if (sh >= 0) {
    const unsigned long long v = static_cast<unsigned long long>(M) << sh;  // < 2^56
    vh = static_cast<uint32_t>(v >> kLimbBits);
    vl = static_cast<uint32_t>(v) & ((1u << kLimbBits) - 1u);
  } else {
    const int r = -sh;
    vh = 0u;
    vl = r < 32 ? (M >> r) : 0u;
    if ((r < 32 ? (M & ((1u << r) - 1u)) : M) != 0u) flags |= kFlagDeep;
  }
  if (vl) flags |= kFlagTail;
  hi = neg ? -static_cast<int>(vh) : static_cast<int>(vh);
  lo = neg ? -static_cast<int>(vl) : static_cast<int>(vl);
}

__device__ __forceinline__ __int128 combine(long long hh, long long hl, long long lh, long long ll) {
  return (static_cast<__int128>(hh) << 56) + ((static_cast<__int128>(hl) + lh) << 28) + static_cast<__int128>(ll);
}

// Per-unit frame. Eq, Es: the exponents of the largest magnitudes; zero: every score is 0 (one side is all
// zeros). qscale, sscale = 2^(27-E): a value's hi limb is trunc(x * scale). qthr, sthr: raw magnitudes
// below these (zero excepted) may have a lower limb; above, a value's least significant bit is at least
// 2^(E-27). narrow: no value of either side is below its threshold, so every lower limb is 0. general: the
// unit takes the general 640-bit path (a non-finite value, or a side whose largest magnitude is below
// 2^-99, where 2^(27-E) is not a float).
struct Frame {
  int Eq, Es;
  bool zero, narrow, general;
  float qscale, sscale;
  uint32_t qthr, sthr;
};

// Shapes of the lane-parallel scorer for a CTA of NT threads: a row of D elements is cut into D/16
// slices, one per thread; the threads of a row are consecutive lanes of one warp.
template <typename T, int D, int NT>
struct Scorer {
  static constexpr int kSPR = D / kSlice;                      // slices (threads) per row
  static constexpr int kRPP = NT / kSPR;                       // rows per pass of the CTA
  static constexpr int kQW = kSlice + 4;                       // words per slice in the q limb tables
  static constexpr int kQRow = kSPR * kQW;                     // words per query head
  static constexpr int kEPV = 16 / static_cast<int>(sizeof(T));  // elements per 16-byte vector
  static constexpr int kVPS = kSlice / kEPV;                   // vectors per slice
  static_assert(D % kSlice == 0 && 32 % kSPR == 0 && NT % 32 == 0, "slice layout");
  // Shared memory of the q limb tables (hi and lo [G][kQRow] int32) and the per-slice lower-limb masks.
  __host__ __device__ static constexpr size_t smem_bytes(int G) {
    return (2 * static_cast<size_t>(G) * kQRow + kSPR) * sizeof(int);
  }
};

// Running magnitude statistics: the largest, and the smallest nonzero (raw bits without the sign).
struct MagStats {
  uint32_t mx, mn;
};
template <typename T>
__device__ __forceinline__ void add_mag(MagStats& s, uint32_t u) {
  const uint32_t m = u & Fmt<T>::kMag;
  s.mx = max(s.mx, m);
  s.mn = min(s.mn, m - 1u) ;  // zero wraps to the largest value: min over nonzero magnitudes, minus one
}
template <typename T>
__device__ __forceinline__ void add_vec(MagStats& s, const uint4& w) {
#pragma unroll
  for (int e = 0; e < 16 / static_cast<int>(sizeof(T)); ++e) add_mag<T>(s, elem_bits<T>(w, e));
}

// The frame from the group's queries qg [G][D] and n summary-key rows (row r at rows + idx[r] * stride,
// or rows + r * stride without idx), reduced over the CTA; every thread returns it. cache receives this
// thread's slice of row tid / kSPR (the scorer's first pass). red: shared [4 * NT/32]; qmask [kSPR] is
// cleared for load_q_limbs (the barrier inside orders the two).
template <typename T, int D, int NT>
__device__ Frame unit_frame(const T* qg, int G, const T* rows, size_t stride, int n, uint32_t* red, int* qmask,
                            int& flags, uint4 (&cache)[Scorer<T, D, NT>::kVPS], const int* idx = nullptr) {
  using S = Scorer<T, D, NT>;
  using F = Fmt<T>;
  constexpr int NW = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  MagStats q{0u, 0xFFFFFFFFu}, sm{0u, 0xFFFFFFFFu};
  if (tid < S::kSPR) qmask[tid] = 0;  // the query limb masks, filled once the frame is known
  for (int v = tid; v < G * D / S::kEPV; v += NT) add_vec<T>(q, reinterpret_cast<const uint4*>(qg)[v]);
  const int j = tid % S::kSPR;
  for (int r = tid / S::kSPR; r < n; r += S::kRPP) {
    const uint4* src = reinterpret_cast<const uint4*>(rows + static_cast<size_t>(idx ? idx[r] : r) * stride +
                                                      j * kSlice);
#pragma unroll
    for (int c = 0; c < S::kVPS; ++c) {
      const uint4 w = src[c];
      if (r < S::kRPP) cache[c] = w;
      add_vec<T>(sm, w);
    }
  }
  uint32_t v0 = __reduce_max_sync(kAll, q.mx), v1 = __reduce_max_sync(kAll, sm.mx);
  uint32_t v2 = __reduce_min_sync(kAll, q.mn), v3 = __reduce_min_sync(kAll, sm.mn);
  if (lane == 0) {
    red[warp] = v0;
    red[NW + warp] = v1;
    red[2 * NW + warp] = v2;
    red[3 * NW + warp] = v3;
  }
  __syncthreads();
  v0 = lane < NW ? red[lane] : 0u;
  v1 = lane < NW ? red[NW + lane] : 0u;
  v2 = lane < NW ? red[2 * NW + lane] : 0xFFFFFFFFu;
  v3 = lane < NW ? red[3 * NW + lane] : 0xFFFFFFFFu;
  const uint32_t qmx = __reduce_max_sync(kAll, v0), smx = __reduce_max_sync(kAll, v1);
  const uint32_t qmn = __reduce_min_sync(kAll, v2) + 1u, smn = __reduce_min_sync(kAll, v3) + 1u;  // 0: none
  Frame f;
  const bool nonfinite = qmx >= F::kInf || smx >= F::kInf;
  if (nonfinite) flags |= kFlagNonFinite;
  f.zero = qmx == 0u || smx == 0u;
  f.Eq = f.zero || nonfinite ? 0 : top_exp<T>(qmx);
  f.Es = f.zero || nonfinite ? 0 : top_exp<T>(smx);
  f.general = nonfinite || (!f.zero && (f.Eq < -99 || f.Es < -99));
  // A normal value with exponent field e has its least significant bit at or above 2^(e - 127 - kMant):
  // at or above 2^(E-27) once e >= E + 100 + kMant. Subnormals always fall below (E >= -99).
  f.qthr = static_cast<uint32_t>(f.Eq + 100 + F::kMant) << F::kMant;
  f.sthr = static_cast<uint32_t>(f.Es + 100 + F::kMant) << F::kMant;
  f.narrow = !f.general && !f.zero && qmn >= f.qthr && smn >= f.sthr;
  f.qscale = f.general || f.zero ? 0.f : __int_as_float((127 + 27 - f.Eq) << 23);
  f.sscale = f.general || f.zero ? 0.f : __int_as_float((127 + 27 - f.Es) << 23);
  return f;
}

// A value as a float (bf16 widens exactly).
template <typename T>
__device__ __forceinline__ float as_f32(uint32_t u) {
  if constexpr (sizeof(T) == 2)
    return __uint_as_float(u << 16);
  else
    return __uint_as_float(u);
}

// The hi limb trunc(x * 2^(27-E)) of a finite value (exact: a power-of-two scale, then a truncation).
template <typename T>
__device__ __forceinline__ int hi_limb(uint32_t u, float scale) {
  return __float2int_rz(as_f32<T>(u) * scale);
}

// 1 when the value is nonzero and its raw magnitude is below thr: it may have a lower limb.
template <typename T>
__device__ __forceinline__ uint32_t maybe_tail(uint32_t u, uint32_t thr) {
  return ((u & Fmt<T>::kMag) - 1u) < thr - 1u ? 1u : 0u;
}

// The group's queries as limb tables in shared memory: qh, ql [G][kQRow] (slice j of head h at
// h * kQRow + j * kQW) and qmask[0] (bit h: head h has a nonzero lower limb; cleared by unit_frame).
// Values below the 56-bit frame set kFlagDeep. Ends with a barrier. Not called for general units.
template <typename T, int D, int NT>
__device__ void load_q_limbs(const T* qg, int G, const Frame& f, int* qh, int* ql, int* qmask, int& flags) {
  using S = Scorer<T, D, NT>;
  const int tid = threadIdx.x;
  for (int v = tid; v < G * D / S::kEPV; v += NT) {
    const uint4 w = reinterpret_cast<const uint4*>(qg)[v];
    const int h = v * S::kEPV / D, c0 = v * S::kEPV % D;
    bool any_lo = false;
#pragma unroll
    for (int e = 0; e < S::kEPV; ++e) {
      const int c = c0 + e;
      const int idx = h * S::kQRow + (c / kSlice) * S::kQW + c % kSlice;
      const uint32_t u = elem_bits<T>(w, e);
      int hi = f.zero ? 0 : hi_limb<T>(u, f.qscale), lo = 0;
      if (!f.zero && maybe_tail<T>(u, f.qthr)) {
        int fl = 0;
        to_limbs<T>(u, f.Eq, hi, lo, fl);
        flags |= fl & kFlagDeep;
        any_lo |= lo != 0;
      }
      qh[idx] = hi;
      ql[idx] = lo;
    }
    if (any_lo) atomicOr(&qmask[0], 1 << h);
  }
  __syncthreads();
}

// Order-preserving unsigned form of a signed 128-bit key (high word's sign bit flipped).
__device__ __forceinline__ void ordered(__int128 v, uint64_t& uh, uint64_t& ul) {
  uh = static_cast<uint64_t>(static_cast<unsigned __int128>(v) >> 64) ^ 0x8000000000000000ull;
  ul = static_cast<uint64_t>(v);
}

// Exact keys of rows [0, n) (row r at rows + idx[r] * stride, or rows + r * stride without idx) against
// query heads [h0, h0 + nh), lane-parallel; not for general units. For
// every live row r, the row's first thread calls emit(r, h, uh, ul) for each head (kMax false), or once
// with the maximum over the heads (kMax true, h = h0). (uh, ul) is the key as an order-preserving
// unsigned 128-bit value: for a narrow unit (0, HH with its sign flipped), S = HH 2^56 exactly; otherwise
// the full int128 S. Every thread must call it. Values below the 56-bit frame set kFlagDeep.
//
// Every value's hi limb comes from the float path. In a unit that is not narrow, a query head with a
// lower limb adds LH = ql . sh (a second dot of the same shape), and a thread whose slice holds values
// that may have a lower limb splits those exactly and adds their HL and LL terms.
template <typename T, int D, int NT, bool kMax, class Emit>
__device__ void score_rows(const T* rows, size_t stride, int n, const Frame& f, const int* qh, const int* ql,
                           const int* qmask, int h0, int nh, int& flags,
                           const uint4 (&cache)[Scorer<T, D, NT>::kVPS], Emit&& emit,
                           const int* idx = nullptr) {
  using S = Scorer<T, D, NT>;
  constexpr uint64_t kSign = 0x8000000000000000ull;
  const int tid = threadIdx.x, j = tid % S::kSPR;
  const uint32_t qheads = f.narrow ? 0u : static_cast<uint32_t>(qmask[0]);  // CTA-uniform
  for (int r0 = 0; r0 < n; r0 += S::kRPP) {
    // a warp whose rows all lie past n is done (later passes start further on); warp-uniform
    if (r0 + (tid & ~31) / S::kSPR >= n) break;
    const int r = r0 + tid / S::kSPR;
    const bool live = r < n;
    const T* src = rows + static_cast<size_t>(live && idx ? idx[r] : (live ? r : 0)) * stride + j * kSlice;
    int sh[kSlice];
    uint32_t tm = 0;  // elements of this slice that may have a lower limb
    {
      uint4 w[S::kVPS];
#pragma unroll
      for (int c = 0; c < S::kVPS; ++c) {
        if (r0 == 0)
          w[c] = live ? cache[c] : make_uint4(0, 0, 0, 0);
        else
          w[c] = live ? reinterpret_cast<const uint4*>(src)[c] : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int c = 0; c < S::kVPS; ++c)
#pragma unroll
        for (int e = 0; e < S::kEPV; ++e) {
          const uint32_t u = elem_bits<T>(w[c], e);
          sh[c * S::kEPV + e] = f.zero ? 0 : hi_limb<T>(u, f.sscale);
          if (!f.narrow) tm |= maybe_tail<T>(u, f.sthr) << (c * S::kEPV + e);
        }
    }
    // warp-uniform: some row slice of this warp may hold a lower limb
    const bool swide = !f.narrow && !f.zero && __any_sync(kAll, tm != 0u);
    __int128 best = 0;
    long long best_hh = 0;
    for (int hb = 0; hb < nh; hb += 4) {
      long long hh[4] = {0, 0, 0, 0}, lh[4] = {0, 0, 0, 0}, hl[4] = {0, 0, 0, 0}, ll[4] = {0, 0, 0, 0};
      const uint32_t qchunk = (qheads >> (h0 + hb)) & 0xFu;  // heads of this chunk with lower limbs
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (hb + c < nh) {
          const int* qhp = qh + (h0 + hb + c) * S::kQRow + j * S::kQW;
#pragma unroll
          for (int t4 = 0; t4 < kSlice; t4 += 4) {
            const int4 a = *reinterpret_cast<const int4*>(qhp + t4);
            hh[c] += static_cast<long long>(a.x) * sh[t4] + static_cast<long long>(a.y) * sh[t4 + 1];
            hh[c] += static_cast<long long>(a.z) * sh[t4 + 2] + static_cast<long long>(a.w) * sh[t4 + 3];
          }
          if ((qchunk >> c) & 1u) {  // LH = ql . sh, a second dot of the same shape
            const int* qlp = ql + (h0 + hb + c) * S::kQRow + j * S::kQW;
#pragma unroll
            for (int t4 = 0; t4 < kSlice; t4 += 4) {
              const int4 a = *reinterpret_cast<const int4*>(qlp + t4);
              lh[c] += static_cast<long long>(a.x) * sh[t4] + static_cast<long long>(a.y) * sh[t4 + 1];
              lh[c] += static_cast<long long>(a.z) * sh[t4 + 2] + static_cast<long long>(a.w) * sh[t4 + 3];
            }
          }
        }
      }
      if (swide) {
        // HL and LL over this slice's values that may have a lower limb (usually none or one), each
        // reloaded (L1) and split exactly; the hi limb equals the float path's
        for (uint32_t m = tm; m; m &= m - 1u) {
          const int t = __ffs(static_cast<int>(m)) - 1;
          int hi = 0, lo = 0, fl = 0;
          to_limbs<T>(raw_at(src, t), f.Es, hi, lo, fl);
          flags |= fl & kFlagDeep;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            if (hb + c < nh) {
              const int at = (h0 + hb + c) * S::kQRow + j * S::kQW + t;
              hl[c] += static_cast<long long>(qh[at]) * lo;
              ll[c] += static_cast<long long>(ql[at]) * lo;
            }
          }
        }
      }
      // sum the row's slices (consecutive lanes); every partial sum stays below 2^63 in magnitude
#pragma unroll
      for (int o = S::kSPR / 2; o > 0; o >>= 1) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          hh[c] += __shfl_xor_sync(kAll, hh[c], o);
          if (qchunk) lh[c] += __shfl_xor_sync(kAll, lh[c], o);
          if (swide) {
            hl[c] += __shfl_xor_sync(kAll, hl[c], o);
            ll[c] += __shfl_xor_sync(kAll, ll[c], o);
          }
        }
      }
      if (j == 0 && live) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (hb + c >= nh) continue;
          if (f.narrow) {
            if constexpr (kMax) {
              if (hb + c == 0 || hh[c] > best_hh) best_hh = hh[c];
            } else {
              emit(r, h0 + hb + c, 0ull, static_cast<uint64_t>(hh[c]) ^ kSign);
            }
          } else {
            const __int128 v = combine(hh[c], hl[c], lh[c], ll[c]);
            if constexpr (kMax) {
              if (hb + c == 0 || v > best) best = v;
            } else {
              uint64_t uh, ul;
              ordered(v, uh, ul);
              emit(r, h0 + hb + c, uh, ul);
            }
          }
        }
      }
    }
    if constexpr (kMax) {
      if (j == 0 && live) {
        uint64_t uh, ul;
        if (f.narrow) {
          uh = 0;
          ul = static_cast<uint64_t>(best_hh) ^ kSign;
        } else {
          ordered(best, uh, ul);
        }
        emit(r, h0, uh, ul);
      }
    }
  }
}

// ------------------------------------------------------------------ general path
// Exact q . s of one row pair as a 640-bit two's-complement integer (digit 0 least significant) in units
// of 2^(2 kMinLe): every product of integer significands added at its absolute bit offset.
template <typename T, int D>
__device__ void big_dot(const T* q, const T* s, uint32_t (&out)[kBigDigits], int& flags) {
  using F = Fmt<T>;
  long long acc[kBigDigits];
#pragma unroll
  for (int i = 0; i < kBigDigits; ++i) acc[i] = 0;
  for (int t = 0; t < D; ++t) {
    uint32_t Mq, Ms;
    int lq, ls;
    bool nq, ns;
    unpack<T>(finite_or_zero<T>(raw_at(q, t), flags), Mq, lq, nq);
    unpack<T>(finite_or_zero<T>(raw_at(s, t), flags), Ms, ls, ns);
    if (Mq == 0u || Ms == 0u) continue;
    const unsigned long long P = static_cast<unsigned long long>(Mq) * Ms;  // < 2^48
    const int off = (lq - F::kMinLe) + (ls - F::kMinLe);                     // <= 506
    const int di = off >> 5, b = off & 31;
    const uint32_t lo = static_cast<uint32_t>(P), hi = static_cast<uint32_t>(P >> 32);
    const uint32_t w0 = lo << b, w1 = __funnelshift_l(lo, hi, b), w2 = b ? hi >> (32 - b) : 0u;
    if (nq != ns) {
      acc[di] -= w0;
      acc[di + 1] -= w1;
      acc[di + 2] -= w2;
    } else {
      acc[di] += w0;
      acc[di + 1] += w1;
      acc[di + 2] += w2;
    }
  }
  long long carry = 0;
#pragma unroll
  for (int i = 0; i < kBigDigits; ++i) {
    const long long v = acc[i] + carry;
    out[i] = static_cast<uint32_t>(v);
    carry = v >> 32;
  }
}

// Sign of a - b for two general-path keys.
__device__ __forceinline__ int big_cmp(const uint32_t* a, const uint32_t* b);

// General-path keys of rows [0, n) (row r at rows + idx[r] * stride, or rows + r * stride without idx),
// written to keys (row r at keys + r * kBigDigits): the maximum over the query heads [h0, h0 + nh) of qg
// of the exact q_h . s_r. Ends with a barrier.
template <typename T, int D, int NT>
__device__ __noinline__ void big_keys(const T* qg, int h0, int nh, const T* rows, size_t stride, int n,
                                      uint32_t* keys, const int* idx = nullptr) {
  int fl = 0;
  for (int r = threadIdx.x; r < n; r += NT) {
    uint32_t best[kBigDigits], cur[kBigDigits];
    const T* row = rows + static_cast<size_t>(idx ? idx[r] : r) * stride;
    for (int h = h0; h < h0 + nh; ++h) {
      big_dot<T, D>(qg + static_cast<size_t>(h) * D, row, cur, fl);
      if (h == h0 || big_cmp(cur, best) > 0)
        for (int i = 0; i < kBigDigits; ++i) best[i] = cur[i];
    }
    for (int i = 0; i < kBigDigits; ++i) keys[static_cast<size_t>(r) * kBigDigits + i] = best[i];
  }
  __syncthreads();
}

// Sign of a - b for two general-path keys.
__device__ __forceinline__ int big_cmp(const uint32_t* a, const uint32_t* b) {
  const int ta = static_cast<int>(a[kBigDigits - 1]), tb = static_cast<int>(b[kBigDigits - 1]);
  if (ta != tb) return ta < tb ? -1 : 1;
  for (int i = kBigDigits - 2; i >= 0; --i)
    if (a[i] != b[i]) return a[i] < b[i] ? -1 : 1;
  return 0;
}

// flag[i] = 1 for the k segments first in (key desc, index asc) over general-path keys (global memory,
// row i at keys + i * kBigDigits). Counting, for any n.
template <int NT>
__device__ __noinline__ void big_rank_select(const uint32_t* keys, int n, int k, int* flag) {
  for (int i = threadIdx.x; i < n; i += NT) {
    const uint32_t* ki = keys + static_cast<size_t>(i) * kBigDigits;
    int beat = 0;
    for (int j = 0; j < n && beat < k; ++j) {
      const int c = big_cmp(keys + static_cast<size_t>(j) * kBigDigits, ki);
      beat += (c > 0) | ((c == 0) & (j < i));
    }
    flag[i] = beat < k ? 1 : 0;
  }
}

// ------------------------------------------------------------------ top-k on 128-bit keys
__device__ __forceinline__ unsigned __int128 u128(uint64_t hi, uint64_t lo) {
  return (static_cast<unsigned __int128>(hi) << 64) | lo;
}
__device__ __forceinline__ unsigned __int128 shr128(unsigned __int128 x, int s) { return s >= 128 ? 0 : x >> s; }

// Exclusive prefix sum of one int per thread over a CTA of NT threads; *total gets the sum.
template <int NT>
__device__ int block_excl_scan(int v, int* total, int* wsum) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kAll, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[w] = x;
  __syncthreads();
  int base = 0, tot = 0;
#pragma unroll
  for (int i = 0; i < NT / 32; ++i) {
    const int s = wsum[i];
    base += i < w ? s : 0;
    tot += s;
  }
  __syncthreads();
  *total = tot;
  return base + x - v;
}

// The radix part of rank_select: 0 < k < n. Most significant digit first, from the highest bit where the
// keys differ; 8-bit digits; stops when the k-th key's bucket is taken whole or at full depth, where equal
// keys go to the lower indices.
template <int NT>
__device__ __noinline__ void radix_top_k(const uint64_t* uh, const uint64_t* ul, int n, int k, int* flag) {
  const int tid = threadIdx.x;
  __shared__ unsigned long long s_mm[4][NT / 32];
  __shared__ int s_hist[256];
  __shared__ int s_sel[3];
  __shared__ int s_wsum[32];
  const int lane = tid & 31, warp = tid >> 5;
  unsigned __int128 mn = ~static_cast<unsigned __int128>(0), mx = 0;
  for (int i = tid; i < n; i += NT) {
    const unsigned __int128 x = u128(uh[i], ul[i]);
    mn = x < mn ? x : mn;
    mx = x > mx ? x : mx;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned __int128 a = u128(__shfl_xor_sync(kAll, static_cast<uint64_t>(mn >> 64), o),
                                     __shfl_xor_sync(kAll, static_cast<uint64_t>(mn), o));
    const unsigned __int128 b = u128(__shfl_xor_sync(kAll, static_cast<uint64_t>(mx >> 64), o),
                                     __shfl_xor_sync(kAll, static_cast<uint64_t>(mx), o));
    mn = a < mn ? a : mn;
    mx = b > mx ? b : mx;
  }
  if (lane == 0) {
    s_mm[0][warp] = static_cast<uint64_t>(mn >> 64);
    s_mm[1][warp] = static_cast<uint64_t>(mn);
    s_mm[2][warp] = static_cast<uint64_t>(mx >> 64);
    s_mm[3][warp] = static_cast<uint64_t>(mx);
  }
  __syncthreads();
  for (int w = 0; w < NT / 32; ++w) {
    const unsigned __int128 a = u128(s_mm[0][w], s_mm[1][w]), b = u128(s_mm[2][w], s_mm[3][w]);
    mn = a < mn ? a : mn;
    mx = b > mx ? b : mx;
  }
  const unsigned __int128 diff = mn ^ mx;
  if (diff == 0) {  // every key equal: the k lowest indices
    for (int i = tid; i < n; i += NT) flag[i] = i < k ? 1 : 0;
    __syncthreads();
    return;
  }
  const uint64_t dh = static_cast<uint64_t>(diff >> 64), dl = static_cast<uint64_t>(diff);
  int pos = dh ? 127 - __clzll(static_cast<long long>(dh)) : 63 - __clzll(static_cast<long long>(dl));
  unsigned __int128 prefix = shr128(mx, pos + 1);  // the bits above pos, shared by every key
  int need = k;
  bool take_all = false;
  while (true) {
    const int width = pos + 1 < 8 ? pos + 1 : 8;
    const int shift = pos + 1 - width;
    const int nb = 1 << width;
    for (int b = tid; b < 256; b += NT) s_hist[b] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += NT) {
      const unsigned __int128 x = u128(uh[i], ul[i]);
      if (shr128(x, pos + 1) == prefix) atomicAdd(&s_hist[static_cast<int>(shr128(x, shift)) & (nb - 1)], 1);
    }
    __syncthreads();
    if (warp == 0) {
      // lane l holds bins nb-1-8l .. nb-8-8l (descending digits)
      int local = 0;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int b = nb - 1 - 8 * lane - c;
        local += b >= 0 ? s_hist[b] : 0;
      }
      int incl = local;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kAll, incl, o);
        if (lane >= o) incl += y;
      }
      const int above = incl - local;
      if (above < need && need <= incl) {
        int cum = above;
        for (int c = 0; c < 8; ++c) {
          const int b = nb - 1 - 8 * lane - c;
          const int h = b >= 0 ? s_hist[b] : 0;
          if (b >= 0 && cum + h >= need) {
            s_sel[0] = b;
            s_sel[1] = cum;
            s_sel[2] = h;
            break;
          }
          cum += h;
        }
      }
    }
    __syncthreads();
    const int D = s_sel[0], above = s_sel[1], cnt = s_sel[2];
    need -= above;
    prefix = (prefix << width) | static_cast<unsigned>(D);
    pos = shift - 1;
    if (cnt == need) {
      take_all = true;
      break;
    }
    if (pos < 0) break;
  }
  // prefix now holds the bits above pos of the k-th key; keys above it are in, keys below are out; keys
  // equal to it are all in (take_all) or, at full depth, the `need` lowest indices among them.
  if (take_all) {
    for (int i = tid; i < n; i += NT) flag[i] = shr128(u128(uh[i], ul[i]), pos + 1) >= prefix ? 1 : 0;
    __syncthreads();
    return;
  }
  const int per = (n + NT - 1) / NT;
  const int i0 = min(n, tid * per), i1 = min(n, i0 + per);
  int eq = 0;
  for (int i = i0; i < i1; ++i) eq += u128(uh[i], ul[i]) == prefix;
  int total;
  int rank = block_excl_scan<NT>(eq, &total, s_wsum);
  for (int i = i0; i < i1; ++i) {
    const unsigned __int128 x = u128(uh[i], ul[i]);
    if (x == prefix) {
      flag[i] = rank < need ? 1 : 0;
      ++rank;
    } else {
      flag[i] = x > prefix ? 1 : 0;
    }
  }
  __syncthreads();
}

// flag[i] = 1 for the k first of n 32-bit keys (the low words of ul) in the order (key desc, index asc);
// any k. Most significant digit first, 8-bit digits from the highest bit where the keys differ, two
// histograms in turn (the next one is cleared while the current one is counted): two barriers a digit.
// Ends with a barrier.
template <int NT>
__device__ __noinline__ void radix_top_k32(const uint64_t* ul, int n, int k, int* flag) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __shared__ int s_hist[2][256];
  __shared__ uint32_t s_mm[2][NT / 32];
  __shared__ int s_sel[3];
  __shared__ int s_wsum[NT / 32];
  if (k <= 0 || k >= n) {
    for (int i = tid; i < n; i += NT) flag[i] = k > 0 ? 1 : 0;
    __syncthreads();
    return;
  }
  auto key = [&](int i) { return static_cast<uint32_t>(ul[i]); };
  auto above_bits = [](uint32_t x, int s) { return s >= 32 ? 0u : x >> s; };
  uint32_t mn = 0xFFFFFFFFu, mx = 0u;
  for (int i = tid; i < n; i += NT) {
    const uint32_t x = key(i);
    mn = min(mn, x);
    mx = max(mx, x);
  }
  mn = __reduce_min_sync(kAll, mn);
  mx = __reduce_max_sync(kAll, mx);
  if (lane == 0) {
    s_mm[0][warp] = mn;
    s_mm[1][warp] = mx;
  }
  for (int b = tid; b < 256; b += NT) s_hist[0][b] = 0;
  __syncthreads();
  mn = __reduce_min_sync(kAll, lane < NT / 32 ? s_mm[0][lane] : 0xFFFFFFFFu);
  mx = __reduce_max_sync(kAll, lane < NT / 32 ? s_mm[1][lane] : 0u);
  if (mn == mx) {  // every key equal: the k lowest indices
    for (int i = tid; i < n; i += NT) flag[i] = i < k ? 1 : 0;
    __syncthreads();
    return;
  }
  int pos = 31 - __clz(static_cast<int>(mn ^ mx));
  uint32_t prefix = above_bits(mx, pos + 1);  // the bits above pos, shared by every key
  int need = k, buf = 0;
  bool take_all = false;
  while (true) {
    const int width = pos + 1 < 8 ? pos + 1 : 8;
    const int shift = pos + 1 - width;
    const int nb = 1 << width;
    for (int i = tid; i < n; i += NT) {
      const uint32_t x = key(i);
      if (above_bits(x, pos + 1) == prefix) atomicAdd(&s_hist[buf][(x >> shift) & (nb - 1)], 1);
    }
    for (int b = tid; b < 256; b += NT) s_hist[buf ^ 1][b] = 0;  // read last before the previous barrier
    __syncthreads();
    if (warp == 0) {
      // lane l holds bins nb-1-8l .. nb-8-8l (descending digits)
      int local = 0;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int b = nb - 1 - 8 * lane - c;
        local += b >= 0 ? s_hist[buf][b] : 0;
      }
      int incl = local;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kAll, incl, o);
        if (lane >= o) incl += y;
      }
      const int above = incl - local;
      if (above < need && need <= incl) {
        int cum = above;
        for (int c = 0; c < 8; ++c) {
          const int b = nb - 1 - 8 * lane - c;
          const int h = b >= 0 ? s_hist[buf][b] : 0;
          if (b >= 0 && cum + h >= need) {
            s_sel[0] = b;
            s_sel[1] = cum;
            s_sel[2] = h;
            break;
          }
          cum += h;
        }
      }
    }
    __syncthreads();
    const int Dg = s_sel[0], above = s_sel[1], cnt = s_sel[2];
    need -= above;
    prefix = (prefix << width) | static_cast<uint32_t>(Dg);
    pos = shift - 1;
    buf ^= 1;
    if (cnt == need) {
      take_all = true;
      break;
    }
    if (pos < 0) break;
  }
  // prefix: the bits above pos of the k-th key. Keys above it are in, keys below it are out; keys equal
  // to it are all in (take_all) or, at full depth, the `need` lowest indices among them.
  if (take_all) {
    for (int i = tid; i < n; i += NT) flag[i] = above_bits(key(i), pos + 1) >= prefix ? 1 : 0;
    __syncthreads();
    return;
  }
  const int per = (n + NT - 1) / NT;
  const int i0 = min(n, tid * per), i1 = min(n, i0 + per);
  int eq = 0;
  for (int i = i0; i < i1; ++i) eq += key(i) == prefix;
  int total;
  int rank = block_excl_scan<NT>(eq, &total, s_wsum);
  for (int i = i0; i < i1; ++i) {
    const uint32_t x = key(i);
    if (x == prefix) {
      flag[i] = rank < need ? 1 : 0;
      ++rank;
    } else {
      flag[i] = x > prefix ? 1 : 0;
    }
  }
  __syncthreads();
}

// flag[i] = 1 for the k first keys in the order (key desc, index asc), keys given as order-preserving
// unsigned 128-bit values (uh, ul) in shared memory; wide = false when every uh is 0. 0 <= k, n >= 1.
template <int NT>
__device__ void rank_select(const uint64_t* uh, const uint64_t* ul, int n, int k, bool wide, int* flag) {
  const int tid = threadIdx.x;
  if (k <= 0 || k >= n) {
    for (int i = tid; i < n; i += NT) flag[i] = k > 0 ? 1 : 0;
    __syncthreads();
    return;
  }
  if (n <= kRadixMinN) {
    // counting: i is selected iff fewer than k keys beat it (greater, or equal with a lower index); P
    // consecutive lanes share segment i, each counting over a stride-P subset of the others
    const int P = n <= NT / 8 ? 8 : (n <= NT / 4 ? 4 : (n <= NT / 2 ? 2 : 1));
    for (int base = 0; base < n * P; base += NT) {
      const int i = (base + tid) / P, part = (base + tid) % P;
      int beat = 0;
      if (i < n) {
        if (wide) {
          const unsigned __int128 ki = u128(uh[i], ul[i]);
          for (int jj = part; jj < n; jj += P) {
            const unsigned __int128 kj = u128(uh[jj], ul[jj]);
            beat += (kj > ki) | ((kj == ki) & (jj < i));
          }
        } else {
          const uint64_t ki = ul[i];
#pragma unroll 4
          for (int jj = part; jj < n; jj += P) {
            const uint64_t kj = ul[jj];
            beat += (kj > ki) | ((kj == ki) & (jj < i));
          }
        }
      }
      for (int o = 1; o < P; o <<= 1) beat += __shfl_xor_sync(kAll, beat, o);
      if (i < n && part == 0) flag[i] = beat < k ? 1 : 0;
    }
    __syncthreads();
    return;
  }
  radix_top_k<NT>(uh, ul, n, k, flag);
}

// ------------------------------------------------------------------ certified fp32 filter
// The exact path above is only needed where an fp32 estimate cannot decide the top-k. Every key is first
// estimated in fp32 with an enclosure that provably contains the exact value; when every selected key's
// lower bound exceeds every other key's upper bound, the fp32 selection is the exact selection.
//
// Error bound (a running bound). A lane sums its 16 or 32 products with fused multiply-adds, and the
// row's slices are added in a shuffle tree of at most 3 levels: at most 135 operations, each
// rounding its exact result once to nearest. Such a rounding changes a result r by at most u |r| + 2^-126
// (u = 2^-24; the second term covers a subnormal result, rounded or flushed to zero), and the errors of
// the operations add up without amplification (every operation takes the previous results as they are),
// so the computed sum a satisfies |a - q.s| <= u R + 2^-118, R = the sum of |r| over every operation that
// led to a. Each lane accumulates R with upward rounding next to its sums (the tree adds the partner's R
// and the new |r|), so the computed R is at least the true one, and eps = u R + 2^-118 rounded up bounds
// the error:
// [a - eps, a + eps] (rounded outward) encloses q . s. The maximum over the group's heads is enclosed
// by the maxima of the bounds. A non-finite estimate or R (an overflow, or a non-finite input) gets
// (-inf, +inf), which no certificate accepts.

__device__ __forceinline__ uint32_t order_bits(float x) {  // order-preserving for finite values and infinities
  const uint32_t b = __float_as_uint(x);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float from_order_bits(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

// Shapes of the estimate for a CTA of NT threads when a lane takes ES consecutive elements of a row.
template <typename T, int D, int NT, int ES>
struct EstShape {
  static constexpr int kEPV = 16 / static_cast<int>(sizeof(T));  // elements per 16-byte word
  static constexpr int kSPR = D / ES;                            // lanes per row
  static constexpr int kRPP = NT / kSPR;                         // rows per pass
  static constexpr int kVPS = ES / kEPV;                         // words per lane and row
  static_assert(D % ES == 0 && 32 % kSPR == 0 && kSPR >= 4 && ES % kEPV == 0, "estimate layout");
};

// The group's queries qg [G][D] in shared memory for estimate_rows, in their own type: qs holds G * D
// values, head h's lane-j slice as kVPS 16-byte words at ((h * kVPS + v) * kSPR + j), so that the lanes
// of a row read consecutive words. Ends with a barrier.
template <typename T, int D, int NT, int ES>
__device__ void load_q_table(const T* qg, int G, uint4* qs) {
  using S = EstShape<T, D, NT, ES>;
  for (int vi = threadIdx.x; vi < G * D / S::kEPV; vi += NT) {
    const int h = vi / (D / S::kEPV), c = vi % (D / S::kEPV);  // word c of head h's row
    qs[(h * S::kVPS + c % S::kVPS) * S::kSPR + c / S::kVPS] = reinterpret_cast<const uint4*>(qg)[vi];
  }
  __syncthreads();
}

// fp32 estimates of every row's key with enclosures, lane-parallel (ES elements of a row per lane, the
// lanes of a row consecutive in one warp): for every live row r, the row's first lane calls
// emit(r, h, mid, lo, hi) for each head of [h0, h0 + nh) (kMax false), or once with the maxima over the
// heads (kMax true, h = h0). lo <= exact q.s <= hi; a non-finite estimate gives (-inf, +inf). The
// queries come from load_q_table's table qs, which is built first when qg is not null (the first pass's
// row loads are issued before it, so both latencies overlap). A pass takes kRPP rows; with ES = 16 the
// next pass's row slices are loaded while the current pass computes. Every thread calls it.
//
// With kMax the slices of a row are summed in a transposed tree: at each of the first two levels a lane
// keeps half of its heads and sends the other half to its partner, which keeps those, so that the lanes
// finish with one head each (two lanes per head when kSPR = 8); the maximum over the heads then takes
// two more levels.
template <typename T, int D, int NT, bool kMax, int ES, class Emit>
__device__ void estimate_rows(const T* qg, int G, uint4* qs, int h0, int nh, const T* rows, size_t stride, int n,
                              Emit&& emit) {
  using S = EstShape<T, D, NT, ES>;
  constexpr int HC = 4;                                // heads per chunk
  constexpr bool kDB = ES == 16;                       // double-buffered row slices
  constexpr float kU = 1.0f / 16777216.0f;             // u = 2^-24
  const float kEpsAbs = __uint_as_float(0x04800000u);  // 2^-118 >= 256 operations x 2^-126
  const int tid = threadIdx.x, j = tid % S::kSPR;
  auto load_slice = [&](int r, uint4 (&w)[S::kVPS]) {
    const uint4* src = reinterpret_cast<const uint4*>(rows + static_cast<size_t>(r < n ? r : 0) * stride + j * ES);
#pragma unroll
    for (int c = 0; c < S::kVPS; ++c) w[c] = r < n ? src[c] : make_uint4(0, 0, 0, 0);
  };
  uint4 sw[S::kVPS];
  load_slice(tid / S::kSPR, sw);
  if (qg) load_q_table<T, D, NT, ES>(qg, G, qs);
  for (int r0 = 0; r0 < n; r0 += S::kRPP) {
    if (r0 + (tid & ~31) / S::kSPR >= n) break;  // warp-uniform: no row of this warp is left
    const int r = r0 + tid / S::kSPR;
    const bool live = r < n;
    if (!kDB && r0 > 0) load_slice(r, sw);
    uint4 nx[kDB ? S::kVPS : 1];  // the next pass's slice, in flight during this one
    if constexpr (kDB) load_slice(r + S::kRPP, nx);
    float xs[ES];
#pragma unroll
    for (int c = 0; c < S::kVPS; ++c)
#pragma unroll
      for (int e = 0; e < S::kEPV; ++e) xs[c * S::kEPV + e] = as_f32<T>(elem_bits<T>(sw[c], e));
    float best_mid = -INFINITY, best_lo = -INFINITY, best_hi = -INFINITY;
    bool bad = false;
    for (int hb = 0; hb < nh; hb += HC) {
      float acc[HC], rb[HC];  // the sum, and the running bound R (rounded up)
#pragma unroll
      for (int c = 0; c < HC; ++c) {
        acc[c] = 0.f;
        rb[c] = 0.f;
        if (hb + c < nh) {
#pragma unroll
          for (int v = 0; v < S::kVPS; ++v) {
            const uint4 qw = qs[((h0 + hb + c) * S::kVPS + v) * S::kSPR + j];
#pragma unroll
            for (int e = 0; e < S::kEPV; ++e) {
              acc[c] = __fmaf_rn(as_f32<T>(elem_bits<T>(qw, e)), xs[v * S::kEPV + e], acc[c]);
              rb[c] = __fadd_ru(rb[c], fabsf(acc[c]));
            }
          }
        }
      }
      if constexpr (kMax) {
        // transposed tree: after the first two levels lane j holds head c1 = 2 * b2 + b1 (b2 = bit
        // kSPR/2 of j, b1 = the next lower bit), summed over the lanes that differ in those bits
        constexpr int o2 = S::kSPR / 2, o1 = S::kSPR / 4;
        const bool up2 = (j & o2) != 0, up1 = (j & o1) != 0;
        float a2[2], r2[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {  // keep heads 2 up2 + i, send heads 2 (1 - up2) + i
          const float sa = up2 ? acc[i] : acc[2 + i], sr = up2 ? rb[i] : rb[2 + i];
          const float ka = up2 ? acc[2 + i] : acc[i], kr = up2 ? rb[2 + i] : rb[i];
          a2[i] = __fadd_rn(ka, __shfl_xor_sync(kAll, sa, o2));
          r2[i] = __fadd_ru(__fadd_ru(kr, __shfl_xor_sync(kAll, sr, o2)), fabsf(a2[i]));
        }
        float a1, r1;
        {
          const float sa = up1 ? a2[0] : a2[1], sr = up1 ? r2[0] : r2[1];
          const float ka = up1 ? a2[1] : a2[0], kr = up1 ? r2[1] : r2[0];
          a1 = __fadd_rn(ka, __shfl_xor_sync(kAll, sa, o1));
          r1 = __fadd_ru(__fadd_ru(kr, __shfl_xor_sync(kAll, sr, o1)), fabsf(a1));
        }
#pragma unroll
        for (int o = S::kSPR / 8; o > 0; o >>= 1) {  // the lanes that still hold the same head (kSPR = 8)
          a1 = __fadd_rn(a1, __shfl_xor_sync(kAll, a1, o));
          r1 = __fadd_ru(__fadd_ru(r1, __shfl_xor_sync(kAll, r1, o)), fabsf(a1));
        }
        const int c1 = (up2 ? 2 : 0) + (up1 ? 1 : 0);
        float mid = a1, lo, hi;
        {
          const float eps = __fmaf_ru(kU, r1, kEpsAbs);
          lo = __fsub_rd(a1, eps);
          hi = __fadd_ru(a1, eps);
          if (!isfinite(a1) || !isfinite(eps)) {
            lo = -INFINITY;
            hi = INFINITY;
            bad = true;
          }
          if (hb + c1 >= nh) mid = lo = hi = -INFINITY;  // a head past the group: not in the maximum
        }
#pragma unroll
        for (int o = o1; o <= o2; o <<= 1) {
          mid = fmaxf(mid, __shfl_xor_sync(kAll, mid, o));
          lo = fmaxf(lo, __shfl_xor_sync(kAll, lo, o));
          hi = fmaxf(hi, __shfl_xor_sync(kAll, hi, o));
        }
        best_mid = fmaxf(best_mid, mid);
        best_lo = fmaxf(best_lo, lo);
        best_hi = fmaxf(best_hi, hi);
      } else {
#pragma unroll
        for (int o = S::kSPR / 2; o > 0; o >>= 1)
#pragma unroll
          for (int c = 0; c < HC; ++c) {
            if (hb + c >= nh) continue;
            acc[c] = __fadd_rn(acc[c], __shfl_xor_sync(kAll, acc[c], o));
            rb[c] = __fadd_ru(__fadd_ru(rb[c], __shfl_xor_sync(kAll, rb[c], o)), fabsf(acc[c]));
          }
#pragma unroll
        for (int c = 0; c < HC; ++c) {
          if (hb + c >= nh) continue;
          const float eps = __fmaf_ru(kU, rb[c], kEpsAbs);
          float lo = __fsub_rd(acc[c], eps), hi = __fadd_ru(acc[c], eps);
          if (!isfinite(acc[c]) || !isfinite(eps)) {
            lo = -INFINITY;
            hi = INFINITY;
          }
          if (j == 0 && live) emit(r, h0 + hb + c, acc[c], lo, hi);
        }
      }
    }
    if constexpr (kMax) {
      bad = __any_sync(kAll, bad);  // any head of the row (lanes of other rows only widen it: no harm)
      if (j == 0 && live) emit(r, h0, best_mid, bad ? -INFINITY : best_lo, bad ? INFINITY : best_hi);
    }
    if constexpr (kDB) {
#pragma unroll
      for (int c = 0; c < S::kVPS; ++c) sw[c] = nx[c];
    }
  }
}

// The top-k of the estimates (ties to the lower index) and its certificate: true when every enclosure is
// finite and Lb = min lo over the selected > Hb = max hi over the others; flag then holds the exact
// selection. ul [n] holds order_bits(mid) (uh [n] zero), written before a barrier. Block-wide; every
// thread gets the answer and (Lb, Hb) (NaN for an empty side). red: shared [3 * NT/32], not used by the
// caller until its next barrier.
template <int NT>
__device__ bool certify_top_k(const float* lo, const float* hi, int n, int k, const uint64_t* uh,
                              const uint64_t* ul, int* flag, uint32_t* red, float& Lb, float& Hb) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t L = 0xFFFFFFFFu, H = 0u, bad = 0u;  // min lo over the selected, max hi over the rest (order bits)
  if (n <= kRadixMinN) {
    // counting, P consecutive lanes per segment (as in rank_select), and the bounds in the same pass
    const int P = n <= NT / 8 ? 8 : (n <= NT / 4 ? 4 : (n <= NT / 2 ? 2 : 1));
    for (int base = 0; base < n * P; base += NT) {
      const int i = (base + tid) / P, part = (base + tid) % P;
      int beat = 0;
      if (i < n) {
        const uint64_t ki = ul[i];
#pragma unroll 4
        for (int jj = part; jj < n; jj += P) {
          const uint64_t kj = ul[jj];
          beat += (kj > ki) | ((kj == ki) & (jj < i));
        }
      }
      for (int o = 1; o < P; o <<= 1) beat += __shfl_xor_sync(kAll, beat, o);
      if (i < n && part == 0) {
        const int f = beat < k ? 1 : 0;
        flag[i] = f;
        const float l = lo[i], h = hi[i];
        bad |= !(isfinite(l) && isfinite(h));
        if (f)
          L = min(L, order_bits(l));
        else
          H = max(H, order_bits(h));
      }
    }
  } else {
    radix_top_k32<NT>(ul, n, k, flag);
    for (int i = tid; i < n; i += NT) {
      const float l = lo[i], h = hi[i];
      bad |= !(isfinite(l) && isfinite(h));
      if (flag[i])
        L = min(L, order_bits(l));
      else
        H = max(H, order_bits(h));
    }
  }
  L = __reduce_min_sync(kAll, L);
  H = __reduce_max_sync(kAll, H);
  bad = __reduce_or_sync(kAll, bad);
  if (lane == 0) {
    red[warp] = L;
    red[NT / 32 + warp] = H;
    red[2 * (NT / 32) + warp] = bad;
  }
  __syncthreads();
  L = __reduce_min_sync(kAll, lane < NT / 32 ? red[lane] : 0xFFFFFFFFu);
  H = __reduce_max_sync(kAll, lane < NT / 32 ? red[NT / 32 + lane] : 0u);
  bad = __reduce_or_sync(kAll, lane < NT / 32 ? red[2 * (NT / 32) + lane] : 0u);
  // k = 0 or k >= n: every flag is already exact; a non-finite input still goes to the exact path
  // (which reports it)
  Lb = L == 0xFFFFFFFFu ? __uint_as_float(0x7FC00000u) : from_order_bits(L);
  Hb = H == 0u ? __uint_as_float(0x7FC00000u) : from_order_bits(H);
  if (bad) return false;
  if (k <= 0 || k >= n) return true;
  return Lb > Hb;  // a float comparison: -0 and +0 do not separate
}


// After a failed certificate: the exact top-k from the exact keys of the uncertain segments only. Lb and
// Hb are certify_top_k's bounds (min lo over the provisional top-k, max hi over the rest).
// - A provisional member with lo > Hb has a key above every non-member's, so fewer than k segments can
//   beat it: it stays in.
// - A non-member with hi < Lb is beaten by all k members: it stays out.
// - The rest U (ascending; every non-finite enclosure is in it) is ranked by exact key within U, ties to
//   the lower index, and its first r = k - (members that stay in) are in. A member of U outranked within
//   U by r others is out: those r have keys above Hb, so they are provisional members, of which U holds
//   exactly r with itself among them, a contradiction unless all k - r stayers outrank it too.
// Returns the unit flags the exact keys raised (kFlagNonFinite, kFlagDeep). Scratch: ulist, uflag [n]
// ints (they may alias lo and hi: those are last read before the first barrier); the keys kh, kl [n];
// the q limb tables qh, ql, qmask; red [4 * NT/32]; s_flags; big (n * kBigDigits words, global).
// kMax: the key of a row is the maximum over heads [h0, h0 + nh) (else nh = 1). Block-wide; ends with a
// barrier after flag is final.
template <typename T, int D, int NT, bool kMax>
__device__ __noinline__ int resolve_top_k(const T* qg, int G, int h0, int nh, const T* rows, size_t stride,
                                          int n, int k, const float* lo, const float* hi, float Lb, float Hb,
                                          int* flag, int* ulist, int* uflag, uint64_t* kh, uint64_t* kl, int* qh,
                                          int* ql, int* qmask, uint32_t* red, int* s_flags, uint32_t* big) {
  using S = Scorer<T, D, NT>;
  __shared__ int s_wsum[NT / 32];
  const int tid = threadIdx.x;
  if (tid == 0) *s_flags = 0;
  // 1. the uncertain segments, and the members that stay in; a contiguous slice per thread (<= 32)
  const int per = (n + NT - 1) / NT;
  const int i0 = min(n, tid * per), i1 = min(n, i0 + per);
  uint32_t um = 0u;
  int stay = 0;
  for (int i = i0; i < i1; ++i) {
    const float l = lo[i], h = hi[i];
    const bool in = flag[i] != 0;
    const bool unc = !(isfinite(l) && isfinite(h)) || (in ? l <= Hb : h >= Lb);
    um |= (unc ? 1u : 0u) << (i - i0);
    stay += in && !unc;
  }
  int total;
  int pos = block_excl_scan<NT>(__popc(um) | (stay << 16), &total, s_wsum) & 0xFFFF;  // n < 2^16
  const int m = total & 0xFFFF, r = k - (total >> 16);
  for (int i = i0; i < i1; ++i)
    if ((um >> (i - i0)) & 1u) ulist[pos++] = i;
  __syncthreads();
  // 2. exact keys of U's rows in a frame of their own (keys of U compare exactly with one another)
  int fl = 0;
  uint4 cache[S::kVPS];
  const Frame fr = unit_frame<T, D, NT>(qg, G, rows, stride, m, red, qmask, fl, cache, ulist);
  if (!fr.general) {
    load_q_limbs<T, D, NT>(qg, G, fr, qh, ql, qmask, fl);
    score_rows<T, D, NT, kMax>(
        rows, stride, m, fr, qh, ql, qmask, h0, nh, fl, cache,
        [&](int j, int, uint64_t uh, uint64_t ulw) {
          kh[j] = uh;
          kl[j] = ulw;
        },
        ulist);
  }
  if (fl) atomicOr(s_flags, fl);
  __syncthreads();
  const int uflags = *s_flags;
  // 3. the first r of U
  if (fr.general || (uflags & kFlagDeep)) {
    big_keys<T, D, NT>(qg, h0, nh, rows, stride, m, big, ulist);
    big_rank_select<NT>(big, m, r, uflag);
    __syncthreads();
  } else {
    rank_select<NT>(kh, kl, m, r, !fr.narrow, uflag);
  }
  for (int j = tid; j < m; j += NT) flag[ulist[j]] = uflag[j];
  __syncthreads();
  return uflags;
}

}  // namespace xk
}  // namespace zr
