// fp64_emu.cuh -- IEEE 754 binary64 addition and multiplication on the
// integer pipes.
//
// GB300 issues FP64 adds, multiplies and FMAs at about 1/70 of its FP32 and
// integer rate, so a sweep doing a few FP64 operations per element is bound
// by the FP64 pipe well below the HBM roof.  The functions here compute the
// correctly rounded (round-to-nearest-even) binary64 sum and product with
// 32/64-bit integer instructions, which run on the full-rate pipes in
// parallel with the FP64 unit, and contain no FP64 instruction at all.  The
// result is bit-identical to a hardware add or multiply for every input
// except that every NaN result is the one quiet NaN 0x7FFFFFFFFFFFFFFF.
//
// Method: the textbook binary floating-point addition (J.-M. Muller et al.,
// "Handbook of Floating-Point Arithmetic", 2nd ed., chapter 7; D. Goldberg,
// "What every computer scientist should know about floating-point
// arithmetic", 1991):
//   1. order the operands by magnitude, so |x| >= |y|;
//   2. place both significands (53 bits, implicit one included) in a 64-bit
//      frame with 10 guard bits below them: X = mx << 10 in [2^62, 2^63);
//   3. shift Y right by the exponent difference d;
//   4. add (same signs) or subtract (opposite signs) the frames;
//   5. normalise so the leading one is bit 63;
//   6. round to nearest, ties to even, at bit 11, and pack sign, exponent
//      and significand (a carry out of the significand on rounding moves
//      into the exponent field by the addition itself).
// Fast path and slow path.  The fast path handles normal operands with
// d < 32 whose result is normal, and drops the bits that step 3 shifts out of
// the frame (only when d > 10).  Dropped bits are less than one unit of the
// frame, i.e. less than 2^-10 of the result's last place, so they can only
// change the rounding when the round field is exactly one half.  That case,
// exact cancellation or a cancellation of 31 bits or more, d >= 32, and all
// non-normal operands and results go to the slow path: the complete
// algorithm with a sticky bit (every bit shifted out OR-ed into bit 0 of the
// frame), subnormals and the IEEE special values, still in integer
// arithmetic.  No hardware FP64 instruction appears anywhere, and the slow
// path is inline code on the bit patterns (a call taking or returning
// doubles was measured to add FP64-pipe instructions to every element).
// The functions are __host__ __device__ so the same code can be checked on
// the CPU against the host's IEEE addition.
#pragma once

#include <stdint.h>

// 1: bits() assembles the pattern from the value's two 32-bit words instead
// of one 64-bit reinterpretation.  The results are the same; the generated
// code differs (the compiler can no longer see a test on the exponent field
// as a test on the double), and which form is faster depends on the kernel,
// so a translation unit chooses before including this header.
#ifndef FVF_EMU_BITS_HILO
#define FVF_EMU_BITS_HILO 0
#endif

#if defined(__CUDACC__)
#define FVF_HD __host__ __device__ __forceinline__
#else
#define FVF_HD inline
#endif

namespace fvf {
namespace emu {

constexpr uint64_t kSign = 0x8000000000000000ull;
constexpr uint64_t kFrac = 0x000FFFFFFFFFFFFFull;
constexpr uint64_t kHidden = 0x0010000000000000ull;

FVF_HD uint64_t bits(double x) {
#if defined(__CUDA_ARCH__) && FVF_EMU_BITS_HILO
    return ((uint64_t)(uint32_t)__double2hiint(x) << 32) | (uint32_t)__double2loint(x);
#elif defined(__CUDA_ARCH__)
    return (uint64_t)__double_as_longlong(x);
#else
    uint64_t u;
    __builtin_memcpy(&u, &x, 8);
    return u;
#endif
}

FVF_HD double from_bits(uint64_t u) {
#if defined(__CUDA_ARCH__)
    return __longlong_as_double((long long)u);
#else
    double x;
    __builtin_memcpy(&x, &u, 8);
    return x;
#endif
}

FVF_HD int clz64(uint64_t x) {
#if defined(__CUDA_ARCH__)
    return __clzll((long long)x);
#else
    return x ? __builtin_clzll(x) : 64;
#endif
}

FVF_HD int clz32(uint32_t x) {
#if defined(__CUDA_ARCH__)
    return __clz((int)x);
#else
    return x ? __builtin_clz(x) : 32;
#endif
}

constexpr uint64_t kInf = 0x7FF0000000000000ull;
// The NaN every NaN-valued sum returns (any NaN is a correct IEEE result;
// this is the quiet NaN the GPU's own FP64 unit produces).
constexpr uint64_t kQuietNaN = 0x7FFFFFFFFFFFFFFFull;

// Complete binary64 addition in integer arithmetic, every input: NaNs and
// infinities by the IEEE rules, signed zeros, subnormal operands (biased
// exponent 0 read as 1 without the implicit one), any exponent difference
// (a sticky bit stands for the bits shifted out of the frame), gradual
// underflow (a result below the normal range is shifted right into the
// subnormal encoding, sticky kept, before rounding) and overflow to
// infinity.
FVF_HD uint64_t add_full_int(uint64_t A, uint64_t B) {
    const uint64_t mA = A & ~kSign, mB = B & ~kSign;
    if (mA > kInf || mB > kInf) return kQuietNaN;
    if (mA == kInf || mB == kInf) {
        if (mA == kInf && mB == kInf && ((A ^ B) & kSign)) return kQuietNaN;  // inf - inf
        return mA == kInf ? A : B;
    }
    const bool swap = mA < mB;
    const uint64_t X = swap ? B : A;             // larger magnitude (its sign wins)
    const uint64_t mx = swap ? mB : mA, my = swap ? mA : mB;
    if (my == 0) return mx == 0 ? (A & B & kSign) : X;   // +0 unless both are -0
    uint32_t ex = (uint32_t)(mx >> 52), ey = (uint32_t)(my >> 52);
    uint64_t fx = mx & kFrac, fy = my & kFrac;
    if (ex) fx |= kHidden; else ex = 1;
    if (ey) fy |= kHidden; else ey = 1;
    fx <<= 10;                                   // <= 2^63
    fy <<= 10;
    const uint32_t d = ex - ey;
    uint64_t al;
    if (d < 64) {
        al = fy >> d;
        al |= (uint64_t)((al << d) != fy);       // sticky
    } else {
        al = 1;
    }
    const bool sub = ((A ^ B) & kSign) != 0;
    uint64_t s = sub ? fx - al : fx + al;
    if (s == 0) return 0;                        // exact cancellation: +0
    const int lz = clz64(s);
    s <<= lz;                                    // leading one at bit 63
    int e = (int)ex + 1 - lz;                    // biased exponent of the result
    if (e < 1) {                                 // below the normal range
        const int sh = 1 - e;
        uint64_t t = sh < 64 ? (s >> sh) : 0;
        t |= (uint64_t)(sh < 64 ? ((t << sh) != s) : (s != 0));
        s = t;
        e = 1;
    }
    uint64_t mant = s >> 11;
    const uint32_t rb = (uint32_t)s & 0x7FFu;    // round bits, sticky jammed in
    mant += (rb + (uint32_t)(mant & 1) + 0x3FFu) >> 11;
    if (e >= 0x7FF) return (X & kSign) | kInf;
    // a carry out of the significand moves into the exponent field (also from
    // the largest subnormal to the smallest normal, and to infinity)
    return (X & kSign) | (((uint64_t)(e - 1) << 52) + mant);
}

// Fast path of a + b (any signs).  Returns false when the slow path is
// needed.
FVF_HD bool add_fast_int(uint64_t A, uint64_t B, uint64_t *out) {
    const uint64_t mA = A & ~kSign, mB = B & ~kSign;
    const bool swap = mA < mB;
    const uint64_t X = swap ? B : A;
    const uint64_t mx = swap ? mB : mA, my = swap ? mA : mB;
    const uint32_t ex = (uint32_t)(mx >> 52), ey = (uint32_t)(my >> 52);
    const uint32_t d = ex - ey;
    const uint64_t fx = ((mx & kFrac) | kHidden) << 10;
    const uint64_t fy = ((my & kFrac) | kHidden) << 10;
    const uint64_t al = fy >> (d & 31);
    const bool sub = ((A ^ B) & kSign) != 0;
    uint64_t s = sub ? fx - al : fx + al;
    // Leading zeros counted in the high word only: a zero high word means a
    // cancellation of 31 or more bits, which the slow path handles.
    const int lz = clz32((uint32_t)(s >> 32));
    s <<= (lz & 31);
    const int e = (int)ex + 1 - lz;
    uint64_t mant = s >> 11;
    const uint32_t rb = (uint32_t)s & 0x7FFu;
    mant += (rb + (uint32_t)(mant & 1) + 0x3FFu) >> 11;
    const bool ok = (ey != 0) & (ex != 0x7FF) & (d < 32) & (lz < 32) & (e > 0) & (e < 0x7FF) &
                    !((d > 10) & (rb == 0x400u));
    *out = (X & kSign) | (((uint64_t)(e - 1) << 52) + mant);
    return ok;
}

// Fast path of a + b for operands of the same sign (no cancellation: the
// leading one ends in bit 62 or 63, so normalisation is a one-bit choice).
FVF_HD bool add_same_sign_fast_int(uint64_t A, uint64_t B, uint64_t *out) {
    const bool swap = A < B;                     // same sign: raw order = magnitude order
    const uint64_t mx = (swap ? B : A) & ~kSign, my = (swap ? A : B) & ~kSign;
    const uint32_t ex = (uint32_t)(mx >> 52), ey = (uint32_t)(my >> 52);
    const uint32_t d = ex - ey;
    const uint64_t fx = ((mx & kFrac) | kHidden) << 10;
    const uint64_t fy = ((my & kFrac) | kHidden) << 10;
    uint64_t s = fx + (fy >> (d & 31));          // [2^62, 2^64)
    const uint32_t carry = (uint32_t)(s >> 63);
    s <<= (carry ^ 1u);                          // leading one at bit 63
    const int e = (int)ex + (int)carry;
    uint64_t mant = s >> 11;
    const uint32_t rb = (uint32_t)s & 0x7FFu;
    mant += (rb + (uint32_t)(mant & 1) + 0x3FFu) >> 11;
    const bool ok = (((A ^ B) & kSign) == 0) & (ey != 0) & (ex != 0x7FF) & (d < 32) &
                    (e < 0x7FF) & !((d > 10) & (rb == 0x400u));
    *out = (A & kSign) | (((uint64_t)(e - 1) << 52) + mant);
    return ok;
}

// Correctly rounded a + b on the integer pipes (bits in, bits out).  The
// slow path is inline and works on the bit patterns only: no call and no
// FP64 value crosses a branch, which on this GPU would cost FP64-pipe
// instructions for every element.
FVF_HD uint64_t add_bits(uint64_t A, uint64_t B) {
    uint64_t r;
    if (!add_fast_int(A, B, &r)) r = add_full_int(A, B);
    return r;
}

FVF_HD uint64_t add_same_sign_bits(uint64_t A, uint64_t B) {
    uint64_t r;
    if (!add_same_sign_fast_int(A, B, &r)) r = add_full_int(A, B);
    return r;
}

FVF_HD double add(double a, double b) { return from_bits(add_bits(bits(a), bits(b))); }

// ---------------------------------------------------------------------------
// ((a + b) + c) + d, each addition correctly rounded, for four normal
// operands of one sign whose exponents span at most 9 binades.  The three
// additions share one 64-bit fixed-point frame instead of aligning,
// normalising and packing three times:
//   * with E the largest biased exponent of the four, an operand of
//     exponent e enters as its 53-bit significand times 2^s,
//     s = 9 - (E - e) in [0, 9], so every operand bit is a frame bit and the
//     frame's unit is 2^(E - 9 - 1075);
//   * the operands are accumulated with integer multiply-adds by 2^s (the
//     low word as a 32 x 32 -> 64-bit product added to the frame, the high
//     word's 21 significand bits times 2^s added to the frame's high word),
//     which issue on the FMA pipe instead of loading the ALU pipe with
//     64-bit shifts and additions;
//   * each partial sum is exact in the frame (operands < 2^62, the rounded
//     partial sums stay below 2^64 - 2^11: the largest case rounds
//     2^64 - 2560 to 2^64 - 2048, so no step carries out of the frame) and
//     is then rounded to its 53 leading bits, ties to even, exactly as the
//     binary64 addition rounds it; a partial sum of two or more operands
//     (each at least 2^52 in the frame) has its leading one at bit 53 or
//     above, so the p = 11 - clz(high word) bits below those 53 number 1
//     to 11;
//   * rounding adds 2^(p-1) - 1 + (the kept part's last bit) and clears the
//     p low bits (round half to even: a remainder of exactly 2^(p-1) moves
//     up only when the kept part is odd); the carry of a round-up stays in
//     the frame;
//   * the packed exponent is E + 2 - clz(high word of the sum): the leading
//     one at bit 63 - z is worth 2^(63 - z + E - 1084).
// The operands' sign bit rides along in the high words: with one sign it
// cancels in the exponent differences and lands back in the sign of the
// result, and the high words order the magnitudes.  PRECONDITION: the four
// operands have one sign (zeros included: +0 with positive operands); the
// caller checks it.  Returns false (and an unspecified value) for a zero or
// subnormal operand, a largest exponent below 2^-1013 or at or above 2^1021
// (so the sum cannot overflow), or a spread of more than 9 binades: with
// E >= 10, every s in [0, 9] implies every operand is normal, and a wider
// spread makes some s wrap below zero.

// a * b + c, 32 x 32 -> 64 bits, as one integer multiply-add
FVF_HD uint64_t mad_wide(uint32_t a, uint32_t b, uint64_t c) {
#if defined(__CUDA_ARCH__)
    uint64_t d;
    asm("mad.wide.u32 %0, %1, %2, %3;" : "=l"(d) : "r"(a), "r"(b), "l"(c));
    return d;
#else
    return (uint64_t)a * b + c;
#endif
}

// frame + significand(hi, lo) * pw, pw = 2^s; the caller's bound keeps the
// true sum below 2^64, so neither part carries out
FVF_HD uint64_t frame_add(uint64_t frame, uint32_t hi, uint32_t lo, uint32_t pw) {
    frame = mad_wide(lo, pw, frame);
    const uint32_t sig_hi = (hi & 0xFFFFFu) | 0x100000u;
    const uint32_t h = sig_hi * pw + (uint32_t)(frame >> 32);
    return ((uint64_t)h << 32) | (uint32_t)frame;
}

FVF_HD uint64_t round53_frame(uint64_t S) {
    // 1..11 (0 only for a single operand at s = 0, which the caller declines)
    const uint32_t p = 11u - (uint32_t)clz32((uint32_t)(S >> 32));
    const uint32_t unit = 1u << p;
    const uint32_t lsb = ((uint32_t)S >> p) & 1u;
    // p <= 11, so the cleared bits lie in the low word: a 32-bit mask (a
    // 64-bit one built from a variable shift cost about 9% of the 2D FP64
    // step on GB300)
    return (S + ((unit >> 1) - 1u + lsb)) & ~(uint64_t)(unit - 1u);
}

// True for +0 and -0.
FVF_HD bool is_zero_bits(uint64_t x) {
    return (((uint32_t)(x >> 32) & 0x7FFFFFFFu) | (uint32_t)x) == 0u;
}

// The sum of N operands of one sign in order, (((X0 + X1) + X2) + ...), in
// one frame.  SH is the largest operand shift: 9 for up to four operands
// (sum < 4 * 2^62 = 2^64), 8 for up to eight (sum < 8 * 2^61); the spread
// limit is SH binades and the smallest accepted largest exponent SH + 1.
// The rounding bound above holds for each: every exact partial sum is at
// most N * (2^(53+SH) - 2^SH) and each rounding adds less than 2^11.
//
// ZSLOT (0 or 1; -1 for none) names one operand of the first pair that may
// be +0 or -0.  X0 + X1 is then the other operand exactly (whatever the
// zero's sign, when the other is not zero), so the zero enters the frame
// with weight 0 and takes its partner's high word for the largest exponent
// (and, at the caller, for the sign test).  The first partial sum is then a
// single operand, leading one at bit 52 + s: the rounding that follows needs
// s >= 1 (p >= 1) and leaves such a value unchanged, so the zero's shift is
// counted as its partner's minus one, which wraps below zero (declines) when
// the partner sits at s = 0.  Used for the cells next to a zero boundary
// face, whose face-side neighbour is the zero.
template <int N, int ZSLOT = -1>
FVF_HD bool sum_one_sign_fast(const uint64_t (&X)[N], uint64_t *out) {
    static_assert(N >= 2 && N <= 8, "frame sized for 2..8 operands");
    static_assert(ZSLOT >= -1 && ZSLOT <= 1, "a zero is tolerated in operand 0 or 1 only");
    constexpr uint32_t SH = N <= 4 ? 9u : 8u;
    uint32_t h[N];
#pragma unroll
    for (int q = 0; q < N; ++q) h[q] = (uint32_t)(X[q] >> 32);
    bool zero = false;
    if constexpr (ZSLOT >= 0) {
        zero = is_zero_bits(X[ZSLOT]);
        if (zero) h[ZSLOT] = h[1 - ZSLOT];
    }
    uint32_t hmax = h[0];
#pragma unroll
    for (int q = 1; q < N; ++q) hmax = hmax > h[q] ? hmax : h[q];
    const uint32_t top = hmax >> 20;                 // sign and largest exponent
    uint32_t pw[N], any = 0;
#pragma unroll
    for (int q = 0; q < N; ++q) {
        uint32_t sq = (h[q] >> 20) - top + SH;       // [0, SH] or wrapped below 0
        if (q == ZSLOT) sq -= (uint32_t)zero;
        any |= sq;
        pw[q] = (q == ZSLOT && zero) ? 0u : 1u << (sq & 15u);
    }
    const bool ok = any < 16u && (hmax & 0x7FFFFFFFu) - ((SH + 1u) << 20) <
                                     0x7FC00000u - ((SH + 1u) << 20);
    uint64_t s = round53_frame(frame_add(frame_add(0, h[0], (uint32_t)X[0], pw[0]), h[1],
                                         (uint32_t)X[1], pw[1]));
#pragma unroll
    for (int q = 2; q < N; ++q) s = round53_frame(frame_add(s, h[q], (uint32_t)X[q], pw[q]));
    const uint32_t z = (uint32_t)clz32((uint32_t)(s >> 32));
    // leading one at bit 63 - z, worth 2^(63 - z + E - SH - 1075); the
    // implicit one at bit 52 adds the last 1 to the exponent field
    *out = ((uint64_t)(top + (10u - SH) - z) << 52) + (s >> (11u - z));
    return ok;
}

// The four-operand form written out: the same arithmetic as
// sum_one_sign_fast<4, ZSLOT> (the host check compares both with the CPU),
// in the form measured on GB300; the template instantiated for four
// operands made the 2D FP64 step 11% slower (0.452 against 0.408 ms per
// 8192^2 step).
template <int ZSLOT = -1>
FVF_HD bool sum4_one_sign_fast(uint64_t A, uint64_t B, uint64_t C, uint64_t D, uint64_t *out) {
    static_assert(ZSLOT >= -1 && ZSLOT <= 1, "a zero is tolerated in operand 0 or 1 only");
    uint32_t ah = (uint32_t)(A >> 32), bh = (uint32_t)(B >> 32);
    const uint32_t ch = (uint32_t)(C >> 32), dh = (uint32_t)(D >> 32);
    bool zero = false;
    if constexpr (ZSLOT == 0) {
        zero = is_zero_bits(A);
        if (zero) ah = bh;
    } else if constexpr (ZSLOT == 1) {
        zero = is_zero_bits(B);
        if (zero) bh = ah;
    }
    const uint32_t m1 = ah > bh ? ah : bh, m2 = ch > dh ? ch : dh, hmax = m1 > m2 ? m1 : m2;
    const uint32_t top = hmax >> 20;                 // sign and largest exponent
    const uint32_t sa = (ah >> 20) - top + 9u - (uint32_t)(ZSLOT == 0 && zero);
    const uint32_t sb = (bh >> 20) - top + 9u - (uint32_t)(ZSLOT == 1 && zero);
    const uint32_t sc = (ch >> 20) - top + 9u, sd = (dh >> 20) - top + 9u;
    const bool ok = (sa | sb | sc | sd) < 16u &&
                    (hmax & 0x7FFFFFFFu) - 0x00A00000u < 0x7FC00000u - 0x00A00000u;
    const uint32_t pa = (ZSLOT == 0 && zero) ? 0u : 1u << (sa & 15u);
    const uint32_t pb = (ZSLOT == 1 && zero) ? 0u : 1u << (sb & 15u);
    uint64_t s = frame_add(frame_add(0, ah, (uint32_t)A, pa), bh, (uint32_t)B, pb);
    s = round53_frame(s);
    s = round53_frame(frame_add(s, ch, (uint32_t)C, 1u << (sc & 15u)));
    s = round53_frame(frame_add(s, dh, (uint32_t)D, 1u << (sd & 15u)));
    const uint32_t z = (uint32_t)clz32((uint32_t)(s >> 32));
    // the implicit one at bit 52 adds the last 1 to the exponent field
    *out = ((uint64_t)(top + 1u - z) << 52) + (s >> (11u - z));
    return ok;
}

// ---------------------------------------------------------------------------
// Multiplication.  The same textbook method (Muller et al., chapter 7): the
// product of the two 53-bit significands, both placed at the top of a 64-bit
// word, is a 128-bit value with its leading one in bit 127 or 126; a one-bit
// normalisation, a sticky bit for the low 64 bits, and the rounding and
// packing of the addition above.  The 64 x 64-bit product is formed from
// four 32 x 32 -> 64-bit products, integer multiply-adds that issue on the
// FMA pipe; measured on GB300, a product costs about 31 ALU-pipe and 15
// FMA-pipe instructions, against about 46 ALU-pipe instructions for a
// same-sign addition.
// ---------------------------------------------------------------------------

// hi:lo = a * b exactly.  Every partial sum stays below 2^64.
FVF_HD void mul_64x64(uint64_t a, uint64_t b, uint64_t *hi, uint64_t *lo) {
    const uint32_t al = (uint32_t)a, ah = (uint32_t)(a >> 32);
    const uint32_t bl = (uint32_t)b, bh = (uint32_t)(b >> 32);
    const uint64_t p0 = (uint64_t)al * bl;
    const uint64_t p1 = (uint64_t)al * bh + (p0 >> 32);
    const uint64_t p2 = (uint64_t)ah * bl + (uint32_t)p1;
    *hi = (uint64_t)ah * bh + (p1 >> 32) + (p2 >> 32);
    *lo = (p2 << 32) | (uint32_t)p0;
}

// Complete binary64 multiplication in integer arithmetic, every input: NaN
// and infinity rules (inf * 0 is NaN), signed zeros, subnormal operands
// (normalised first), gradual underflow with a sticky bit, overflow to
// infinity.
FVF_HD uint64_t mul_full_int(uint64_t A, uint64_t B) {
    const uint64_t sgn = (A ^ B) & kSign;
    const uint64_t mA = A & ~kSign, mB = B & ~kSign;
    if (mA > kInf || mB > kInf) return kQuietNaN;
    if (mA == kInf || mB == kInf) return (mA == 0 || mB == 0) ? kQuietNaN : (sgn | kInf);
    if (mA == 0 || mB == 0) return sgn;
    int ea = (int)(mA >> 52), eb = (int)(mB >> 52);
    uint64_t fa = mA & kFrac, fb = mB & kFrac;
    if (ea) {
        fa |= kHidden;
    } else {                                     // subnormal: leading one up to bit 52
        const int sh = clz64(fa) - 11;
        fa <<= sh;
        ea = 1 - sh;
    }
    if (eb) {
        fb |= kHidden;
    } else {
        const int sh = clz64(fb) - 11;
        fb <<= sh;
        eb = 1 - sh;
    }
    uint64_t hi, lo;
    mul_64x64(fa << 11, fb << 11, &hi, &lo);     // in [2^126, 2^128)
    const uint32_t c = (uint32_t)(hi >> 63);
    if (!c) {                                    // leading one to bit 127
        hi = (hi << 1) | (lo >> 63);
        lo <<= 1;
    }
    uint64_t s = hi | (uint64_t)(lo != 0);       // sticky
    int e = ea + eb - 1023 + (int)c;             // biased exponent of the result
    if (e < 1) {                                 // below the normal range
        const int sh = 1 - e;
        uint64_t t = sh < 64 ? (s >> sh) : 0;
        t |= (uint64_t)(sh < 64 ? ((t << sh) != s) : (s != 0));
        s = t;
        e = 1;
    }
    uint64_t mant = s >> 11;
    const uint32_t rb = (uint32_t)s & 0x7FFu;
    mant += (rb + (uint32_t)(mant & 1) + 0x3FFu) >> 11;
    if (e >= 0x7FF) return sgn | kInf;
    return sgn | (((uint64_t)(e - 1) << 52) + mant);
}

// A factor shared by many products (a diffusion or stage coefficient for a
// whole sweep, an inverse spacing for a cell's variables): its significand
// placed at the top of a 64-bit word and its exponent, prepared once.  `fast` is 0 when the factor is zero, subnormal, infinite or NaN;
// every product then takes the complete algorithm.
struct MulConst {
    uint64_t bits;   // the factor's bit pattern
    uint64_t k;      // significand << 11, in [2^63, 2^64)
    uint64_t sign;   // its sign bit
    int32_t adj;     // biased exponent - 1023
    uint32_t fast;
};

// The factor's fields are taken from its two 32-bit words: built from the
// 64-bit pattern, the range test below was measured to cost one FP64-pipe
// instruction per call on GB300 (the compiler may turn a test on a double's
// exponent field into a floating-point comparison).
FVF_HD MulConst mul_const(double alpha) {
#if defined(__CUDA_ARCH__)
    const uint32_t hi = (uint32_t)__double2hiint(alpha), lo = (uint32_t)__double2loint(alpha);
#else
    const uint64_t b = bits(alpha);
    const uint32_t hi = (uint32_t)(b >> 32), lo = (uint32_t)b;
#endif
    MulConst m;
    const uint32_t e = (hi >> 20) & 0x7FFu;
    m.bits = ((uint64_t)hi << 32) | lo;
    m.k = ((uint64_t)((hi & 0xFFFFFu) | 0x100000u) << 43) | ((uint64_t)lo << 11);
    m.sign = (uint64_t)(hi & 0x80000000u) << 32;
    m.adj = (int32_t)e - 1023;
    m.fast = (e - 1u) < 2046u;
    return m;
}

// Fast path of t * alpha: t normal and the result normal (before rounding),
// which leaves no special case.  The sticky bit from the low product half
// makes every rounding exact, ties included.
FVF_HD bool mul_const_fast_int(uint64_t T, const MulConst &m, uint64_t *out) {
    const uint32_t th = (uint32_t)(T >> 32), tl = (uint32_t)T;
    const uint32_t et = (th >> 20) & 0x7FFu;
    // the significand with its implicit one, shifted to the top of the word
    const uint64_t ft = ((uint64_t)(th | 0x00100000u) << 43) | ((uint64_t)tl << 11);
    uint64_t hi, lo;
    mul_64x64(ft, m.k, &hi, &lo);
    const uint32_t c = (uint32_t)(hi >> 63);
    const uint64_t s = hi << (c ^ 1u);
    const int e = (int)et + m.adj + (int)c;
    uint64_t mant = s >> 11;
    const uint32_t rb = ((uint32_t)s & 0x7FFu) | (uint32_t)(lo != 0);
    mant += (rb + (uint32_t)(mant & 1) + 0x3FFu) >> 11;
    *out = ((T & kSign) ^ m.sign) | (((uint64_t)(e - 1) << 52) + mant);
    return m.fast & ((et - 1u) < 2046u) & ((uint32_t)(e - 1) < 2046u);
}

FVF_HD uint64_t mul_const_bits(uint64_t T, const MulConst &m) {
    uint64_t r;
    if (!mul_const_fast_int(T, m, &r)) r = mul_full_int(T, m.bits);
    return r;
}

FVF_HD double mul(double a, double b) { return from_bits(mul_full_int(bits(a), bits(b))); }

// Fastest when a and b have the same sign; correct for any operands.
FVF_HD double add_same_sign(double a, double b) {
    return from_bits(add_same_sign_bits(bits(a), bits(b)));
}

}  // namespace emu
}  // namespace fvf
