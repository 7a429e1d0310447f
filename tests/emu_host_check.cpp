// Host check of the integer-pipe binary64 addition and multiplication
// (fp64_emu.cuh): every sum and product must be bit-identical to the host
// CPU's IEEE 754 operation (round to nearest even), and so must the
// fixed-point sum of four operands, ((a + b) + c) + d, wherever its fast
// form accepts the operands, and the six-operand sum of the 3D update with
// and without a zero in its first pair (and the four-operand sum with such
// a zero).  Built with -O2 -ffp-contract=off; prints "mismatches N cases M
// sum4_taken T sum6_taken U sum6z_taken Z sum4z_taken Y".
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "../finite_volume_field_gb300/csrc/fp64_emu.cuh"

using namespace fvf::emu;

static uint64_t sm_state = 0x243F6A8885A308D3ull;
static uint64_t next_u64() {  // SplitMix64 (Steele, Lea, Flood 2014)
    uint64_t z = (sm_state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static double native_add(double a, double b) {
    volatile double x = a, y = b;
    volatile double r = x + y;
    return r;
}

static double native_mul(double a, double b) {
    volatile double x = a, y = b;
    volatile double r = x * y;
    return r;
}

static uint64_t mismatches = 0, cases = 0;

static bool is_nan(uint64_t x) { return ((x >> 52) & 0x7FF) == 0x7FF && (x & kFrac); }

static void report(const char *what, uint64_t A, uint64_t B, uint64_t got, uint64_t want) {
    if (got == want || (is_nan(got) && is_nan(want))) return;
    if (mismatches < 10)
        std::printf("%s mismatch: %016llx, %016llx -> got %016llx want %016llx\n", what,
                    (unsigned long long)A, (unsigned long long)B, (unsigned long long)got,
                    (unsigned long long)want);
    ++mismatches;
}

// a * b by the complete algorithm, and by the fixed-factor fast path (with
// its fallback) with either operand as the fixed factor
static void check_mul(uint64_t A, uint64_t B) {
    const double a = from_bits(A), b = from_bits(B);
    const uint64_t want = bits(native_mul(a, b));
    ++cases;
    report("mul full", A, B, mul_full_int(A, B), want);
    report("mul", A, B, bits(mul(a, b)), want);
    report("mul const", A, B, mul_const_bits(A, mul_const(b)), want);
    report("mul const swapped", B, A, mul_const_bits(B, mul_const(a)), want);
    uint64_t fast;
    if (mul_const_fast_int(A, mul_const(b), &fast)) report("mul fast", A, B, fast, want);
}

static uint64_t sum4_taken = 0;

// ((A + B) + C) + D: the fixed-point form where it accepts the operands
// (operands of one sign: its precondition).
static void check_sum4(uint64_t A, uint64_t B, uint64_t C, uint64_t D) {
    uint64_t got;
    if (((A ^ B) | (A ^ C) | (A ^ D)) & kSign) return;
    const uint64_t X[4] = {A, B, C, D};
    uint64_t tgot;
    const bool tok = sum_one_sign_fast<4>(X, &tgot);
    if (!sum4_one_sign_fast(A, B, C, D, &got)) {
        if (tok) {                               // the two forms must agree
            if (mismatches < 10) std::printf("sum4 forms disagree on acceptance\n");
            ++mismatches;
        }
        return;
    }
    if (!tok || tgot != got) {
        if (mismatches < 10) std::printf("sum4 forms disagree\n");
        ++mismatches;
    }
    ++sum4_taken;
    ++cases;
    const double want = native_add(native_add(native_add(from_bits(A), from_bits(B)), from_bits(C)),
                                   from_bits(D));
    if (got != bits(want)) {
        if (mismatches < 10)
            std::printf("sum4 %016llx %016llx %016llx %016llx: got %016llx want %016llx\n",
                        (unsigned long long)A, (unsigned long long)B, (unsigned long long)C,
                        (unsigned long long)D, (unsigned long long)got, (unsigned long long)bits(want));
        ++mismatches;
    }
}

static uint64_t sum6_taken = 0;

// (((((X0 + X1) + X2) + X3) + X4) + X5): the six-operand frame where it
// accepts the operands (one sign: its precondition).
static void check_sum6(const uint64_t (&X)[6]) {
    for (int q = 1; q < 6; ++q)
        if ((X[q] ^ X[0]) & kSign) return;
    uint64_t got;
    if (!sum_one_sign_fast<6>(X, &got)) return;
    ++sum6_taken;
    ++cases;
    double want = from_bits(X[0]);
    for (int q = 1; q < 6; ++q) want = native_add(want, from_bits(X[q]));
    if (got != bits(want)) {
        if (mismatches < 10)
            std::printf("sum6 %016llx ... %016llx: got %016llx want %016llx\n", (unsigned long long)X[0],
                        (unsigned long long)X[5], (unsigned long long)got, (unsigned long long)bits(want));
        ++mismatches;
    }
}

static uint64_t make(uint64_t sign, uint64_t exp, uint64_t frac) {
    return (sign << 63) | ((exp & 0x7FF) << 52) | (frac & kFrac);
}

static uint64_t sum6z_taken = 0;

// The same sum with a zero tolerated in operand ZSLOT (0 or 1): the caller's
// sign test takes the partner's sign for a zero there.  Where the form
// accepts a set without a zero in the slot it must also agree with the
// plain form.
template <int ZSLOT>
static void check_sum6_zero_slot(const uint64_t (&X)[6]) {
    uint64_t h[6];
    for (int q = 0; q < 6; ++q) h[q] = X[q];
    if (is_zero_bits(X[ZSLOT])) h[ZSLOT] = X[1 - ZSLOT];
    for (int q = 1; q < 6; ++q)
        if ((h[q] ^ h[0]) & kSign) return;
    uint64_t got;
    if (!sum_one_sign_fast<6, ZSLOT>(X, &got)) return;
    ++cases;
    if (is_zero_bits(X[ZSLOT])) ++sum6z_taken;
    double want = from_bits(X[0]);
    for (int q = 1; q < 6; ++q) want = native_add(want, from_bits(X[q]));
    if (got != bits(want)) {
        if (mismatches < 10)
            std::printf("sum6 zero slot %d %016llx %016llx ... %016llx: got %016llx want %016llx\n", ZSLOT,
                        (unsigned long long)X[0], (unsigned long long)X[1], (unsigned long long)X[5],
                        (unsigned long long)got, (unsigned long long)bits(want));
        ++mismatches;
    }
}

static uint64_t sum4z_taken = 0;

// The four-operand forms with a zero tolerated in operand ZSLOT: the
// written-out form and the template must agree on acceptance and value.
template <int ZSLOT>
static void check_sum4_zero_slot(const uint64_t (&X)[6]) {
    uint64_t h[4];
    for (int q = 0; q < 4; ++q) h[q] = X[q];
    if (is_zero_bits(X[ZSLOT])) h[ZSLOT] = X[1 - ZSLOT];
    for (int q = 1; q < 4; ++q)
        if ((h[q] ^ h[0]) & kSign) return;
    const uint64_t Y[4] = {X[0], X[1], X[2], X[3]};
    uint64_t got, tgot;
    const bool ok = sum4_one_sign_fast<ZSLOT>(X[0], X[1], X[2], X[3], &got);
    const bool tok = sum_one_sign_fast<4, ZSLOT>(Y, &tgot);
    if (ok != tok || (ok && got != tgot)) {
        if (mismatches < 10) std::printf("sum4 zero-slot forms disagree\n");
        ++mismatches;
    }
    if (!ok) return;
    ++cases;
    if (is_zero_bits(X[ZSLOT])) ++sum4z_taken;
    const double want = native_add(native_add(native_add(from_bits(X[0]), from_bits(X[1])), from_bits(X[2])),
                                   from_bits(X[3]));
    if (got != bits(want)) {
        if (mismatches < 10)
            std::printf("sum4 zero slot %d %016llx %016llx %016llx %016llx: got %016llx want %016llx\n", ZSLOT,
                        (unsigned long long)X[0], (unsigned long long)X[1], (unsigned long long)X[2],
                        (unsigned long long)X[3], (unsigned long long)got, (unsigned long long)bits(want));
        ++mismatches;
    }
}

template <int ZSLOT>
static void check_zero_slot(const uint64_t (&X)[6]) {
    check_sum6_zero_slot<ZSLOT>(X);
    check_sum4_zero_slot<ZSLOT>(X);
}

// Sets for the zero-slot forms (four operands: the first four of each set): the slot set to +0 or -0 and its partner
// at every shift the frame can give it (including s = 0, which the form
// must decline, and beyond), zero or subnormal partners, a partner of the
// other sign, smoothed-field values with a zero face neighbour, equal
// values and ties, and largest exponents near both limits.
template <int ZSLOT>
static void zero_slot_cases(long n) {
    constexpr int P = 1 - ZSLOT;
    for (long i = 0; i < n; ++i) {
        uint64_t X[6];
        const uint64_t sg = next_u64() & 1, e0 = 1 + next_u64() % 2046;
        const int spread = (int)(next_u64() % 11);
        for (auto &x : X) {
            int64_t e = (int64_t)e0 - (int64_t)(next_u64() % (spread + 1));
            e = e < 0 ? 0 : e;
            const uint64_t f = (next_u64() & 1) ? next_u64() : next_u64() & ~((1ull << (next_u64() % 53)) - 1);
            x = make(sg, (uint64_t)e, f);
        }
        check_zero_slot<ZSLOT>(X);
        X[ZSLOT] = make(next_u64() & 1, 0, 0);
        check_zero_slot<ZSLOT>(X);
        X[2] = make(sg, e0, next_u64());
        for (uint64_t below = 6; below <= 11; ++below) {
            X[P] = make(sg, e0 >= below ? e0 - below : 0, next_u64());
            check_zero_slot<ZSLOT>(X);
        }
        X[P] = make(next_u64() & 1, 0, (next_u64() & 1) ? 0 : next_u64());
        check_zero_slot<ZSLOT>(X);
        X[P] = make(sg ^ 1, e0, next_u64());
        check_zero_slot<ZSLOT>(X);
        for (auto &x : X) x = bits((double)(next_u64() >> 11) * 0x1p-53);
        X[ZSLOT] = 0;
        check_zero_slot<ZSLOT>(X);
        const uint64_t t = make(sg, 1 + next_u64() % 2046, (next_u64() & 1) ? kFrac : (next_u64() & 0xFFF0000000000ull));
        for (auto &x : X) x = t;
        X[ZSLOT] = make(next_u64() & 1, 0, 0);
        check_zero_slot<ZSLOT>(X);
        for (auto &x : X) x = make(sg, e0 + next_u64() % 2, (next_u64() & 1) ? 1 : (1ull << 51) | 1);
        X[ZSLOT] = make(sg, 0, 0);
        check_zero_slot<ZSLOT>(X);
        for (auto &x : X) x = make(sg, (next_u64() & 1) ? 2037 + next_u64() % 10 : 5 + next_u64() % 10, next_u64());
        X[ZSLOT] = make(sg, 0, 0);
        check_zero_slot<ZSLOT>(X);
    }
}

static void check(uint64_t A, uint64_t B) {
    const double a = from_bits(A), b = from_bits(B);
    const uint64_t want = bits(native_add(a, b));
    const uint64_t got = bits(add(a, b));
    const bool nan = ((want >> 52) & 0x7FF) == 0x7FF && (want & kFrac);
    ++cases;
    if (got != want && !(nan && ((got >> 52) & 0x7FF) == 0x7FF && (got & kFrac))) {
        if (mismatches < 10)
            std::printf("add mismatch: %016llx + %016llx -> got %016llx want %016llx\n",
                        (unsigned long long)A, (unsigned long long)B, (unsigned long long)got,
                        (unsigned long long)want);
        ++mismatches;
    }
    if (((A ^ B) >> 63) == 0) {
        const uint64_t got2 = bits(add_same_sign(a, b));
        if (got2 != want && !nan) {
            if (mismatches < 10)
                std::printf("same-sign mismatch: %016llx + %016llx -> got %016llx want %016llx\n",
                            (unsigned long long)A, (unsigned long long)B,
                            (unsigned long long)got2, (unsigned long long)want);
            ++mismatches;
        }
    }
    // the complete integer algorithm on its own (the slow path)
    const uint64_t full = add_full_int(A, B);
    if (full != want && !(nan && ((full >> 52) & 0x7FF) == 0x7FF && (full & kFrac))) {
        if (mismatches < 10)
            std::printf("full mismatch: %016llx + %016llx -> got %016llx want %016llx\n",
                        (unsigned long long)A, (unsigned long long)B, (unsigned long long)full,
                        (unsigned long long)want);
        ++mismatches;
    }
    // the other operand order must give the same bits (NaNs: any NaN)
    const uint64_t swapped = bits(add(b, a));
    if (swapped != got && !nan) {
        if (mismatches < 10)
            std::printf("order mismatch: %016llx + %016llx -> %016llx vs %016llx\n",
                        (unsigned long long)A, (unsigned long long)B, (unsigned long long)got,
                        (unsigned long long)swapped);
        ++mismatches;
    }
}


int main(int argc, char **argv) {
    const long n = argc > 1 ? std::atol(argv[1]) : 1000000;
    // 1. uniformly random bit patterns
    for (long i = 0; i < n; ++i) check(next_u64(), next_u64());
    // 2. exponents within 70 of each other, random signs and fractions
    for (long i = 0; i < 4 * n; ++i) {
        const uint64_t e = 1 + next_u64() % 2046;
        const int64_t de = (int64_t)(next_u64() % 141) - 70;
        int64_t e2 = (int64_t)e + de;
        if (e2 < 0) e2 = 0;
        if (e2 > 2047) e2 = 2047;
        check(make(next_u64() & 1, e, next_u64()), make(next_u64() & 1, (uint64_t)e2, next_u64()));
    }
    // 3. cancellation: opposite signs, nearly equal magnitudes
    for (long i = 0; i < n; ++i) {
        const uint64_t A = make(0, 1 + next_u64() % 2046, next_u64());
        const int64_t k = (int64_t)(next_u64() % 2049) - 1024;
        uint64_t B = (A + (uint64_t)k) | kSign;
        if (((B >> 52) & 0x7FF) == 0x7FF) B = A | kSign;
        check(A, B);
        check(A, (A ^ kSign) + (next_u64() % 4));
    }
    // 4. ties and near-ties: y is a power of two around half an ulp of x
    for (long i = 0; i < n; ++i) {
        const uint64_t ex = 60 + next_u64() % 1900;
        const uint64_t A = make(next_u64() & 1, ex, next_u64() & ((next_u64() & 1) ? ~0ull : ~7ull));
        const uint64_t ey = ex - 52 - (next_u64() % 4);
        const uint64_t B = make(next_u64() & 1, ey, (next_u64() & 1) ? 0 : next_u64() % 3);
        check(A, B);
    }
    // 5. the ends of the exponent range: subnormal results, overflow
    for (long i = 0; i < n / 4; ++i) {
        check(make(next_u64() & 1, next_u64() % 4, next_u64()), make(next_u64() & 1, next_u64() % 4, next_u64()));
        check(make(next_u64() & 1, 2043 + next_u64() % 5, next_u64()),
              make(next_u64() & 1, 2040 + next_u64() % 8, next_u64()));
    }
    // 6. gradual underflow: subnormal sums and differences of small normals
    for (long i = 0; i < n; ++i) {
        const uint64_t ea = next_u64() % 60, eb = ea + (next_u64() % 5) - 2;
        check(make(next_u64() & 1, ea, next_u64()), make(next_u64() & 1, eb & 0x7FF, next_u64()));
        const uint64_t A = make(0, 1 + next_u64() % 54, next_u64());
        check(A, (A + (next_u64() % 4096) - 2048) | kSign);
    }
    // 7. special values against everything
    const uint64_t specials[] = {0, kSign, 1, kSign | 1, kHidden, kHidden - 1, 0x7FEFFFFFFFFFFFFFull,
                                 0xFFEFFFFFFFFFFFFFull, 0x7FF0000000000000ull, 0xFFF0000000000000ull,
                                 0x7FF8000000000000ull, 0x7FF4000000000001ull, 0x3FF0000000000000ull,
                                 0xBFF0000000000000ull, 0x3CA0000000000000ull, 0x3CB0000000000000ull};
    const int ns = sizeof(specials) / sizeof(specials[0]);
    for (int i = 0; i < ns; ++i)
        for (int j = 0; j < ns; ++j) check(specials[i], specials[j]);
    for (long i = 0; i < n / 10; ++i)
        for (int j = 0; j < ns; ++j) check(specials[j], next_u64());
    // products: random patterns, exponents that put the product anywhere from
    // deep underflow to overflow, ties (significands with few bits), subnormal
    // operands, the diffusion's own factors (0 < alpha <= 1/4, t of any size)
    for (long i = 0; i < n; ++i) check_mul(next_u64(), next_u64());
    for (long i = 0; i < 2 * n; ++i) {
        const uint64_t ea = next_u64() % 2048;
        const int64_t target = (int64_t)(next_u64() % 2300) - 130;   // biased result exponent
        int64_t eb = target + 1023 - (int64_t)ea;
        if (eb < 0) eb = next_u64() % 3;
        if (eb > 2047) eb = 2047 - next_u64() % 3;
        check_mul(make(next_u64() & 1, ea, next_u64()), make(next_u64() & 1, (uint64_t)eb, next_u64()));
    }
    for (long i = 0; i < n; ++i) {
        // significands with at most 26 + 27 significant bits: exact products and halfway cases
        const uint64_t fa = next_u64() & (kFrac & ~((1ull << (next_u64() % 53)) - 1));
        const uint64_t fb = next_u64() & (kFrac & ~((1ull << (next_u64() % 53)) - 1));
        check_mul(make(next_u64() & 1, 1 + next_u64() % 2046, fa), make(next_u64() & 1, 1 + next_u64() % 2046, fb));
        check_mul(make(next_u64() & 1, 0, next_u64()), make(next_u64() & 1, next_u64() % 2048, next_u64()));
    }
    for (long i = 0; i < n; ++i) {
        const double alpha = 0.25 * (double)(next_u64() >> 11) * 0x1p-53;
        check_mul(next_u64(), bits(alpha));
        check_mul(make(next_u64() & 1, 900 + next_u64() % 250, next_u64()), bits(alpha));
        check_mul(bits(0.1), make(next_u64() & 1, next_u64() % 2048, next_u64()));
    }
    for (int i = 0; i < ns; ++i)
        for (int j = 0; j < ns; ++j) check_mul(specials[i], specials[j]);
    for (long i = 0; i < n / 10; ++i)
        for (int j = 0; j < ns; ++j) check_mul(specials[j], next_u64());
    // four-operand sums: one sign, exponents within 10 of a random centre
    // (spreads of 9 and 10 binades, zeros and subnormals near the bottom,
    // results near overflow at the top); significands with few bits (ties
    // in every partial sum); all-ones significands at spreads 0..9 (the
    // largest frame values); the diffusion's own values (uniform [0, 1),
    // products of [0.25, 0.75) and their negatives)
    for (long i = 0; i < n; ++i) {
        const uint64_t sg = next_u64() & 1, e0 = 1 + next_u64() % 2046;
        auto g = [&]() {
            int64_t e = (int64_t)e0 + (int64_t)(next_u64() % 21) - 10;
            e = e < 0 ? 0 : (e > 2047 ? 2047 : e);
            return make(sg, (uint64_t)e, next_u64());
        };
        const uint64_t a = g(), b = g(), c = g(), d = g();
        check_sum4(a, b, c, d);
    }
    for (long i = 0; i < n; ++i) {
        const uint64_t sg = next_u64() & 1, e0 = 1 + next_u64() % 2046;
        auto g = [&]() {
            int64_t e = (int64_t)e0 + (int64_t)(next_u64() % 3) - 1;
            e = e < 0 ? 0 : (e > 2047 ? 2047 : e);
            const uint64_t f = (next_u64() & 1) ? next_u64() : next_u64() & ~((1ull << (next_u64() % 53)) - 1);
            return make(sg, (uint64_t)e, f);
        };
        const uint64_t a = g(), b = g(), c = g(), d = g();
        check_sum4(a, b, c, d);
    }
    for (long i = 0; i < n; ++i) {
        const uint64_t sg = next_u64() & 1, e0 = 1 + next_u64() % 2040;
        auto g = [&]() {
            const uint64_t f = (next_u64() & 1) ? kFrac : (next_u64() & 0xFFF0000000000ull);
            return make(sg, e0 + next_u64() % 10, f);
        };
        const uint64_t a = g(), b = g(), c = g(), d = g();
        check_sum4(a, b, c, d);
        const uint64_t top = make(sg, 2030 + next_u64() % 18, kFrac - next_u64() % 8);
        check_sum4(top, top, top, top);
    }
    for (long i = 0; i < n; ++i) {
        auto u = [&]() { return bits((double)(next_u64() >> 11) * 0x1p-53); };
        const uint64_t a = u(), b = u(), c = u(), d = u();
        check_sum4(a, b, c, d);
        auto v = [&]() { return bits(-(0.25 + 0.5 * (double)(next_u64() >> 11) * 0x1p-53)); };
        const uint64_t e = v(), f = v(), g = v(), h = v();
        check_sum4(e, f, g, h);
    }
    // six-operand sums (the 3D update's neighbours): the same kinds of cases
    // with the 8-binade limit of the six-operand frame
    for (long i = 0; i < n; ++i) {
        const uint64_t sg = next_u64() & 1, e0 = 1 + next_u64() % 2046;
        uint64_t X[6];
        for (auto &x : X) {
            int64_t e = (int64_t)e0 + (int64_t)(next_u64() % 19) - 9;
            e = e < 0 ? 0 : (e > 2047 ? 2047 : e);
            x = make(sg, (uint64_t)e, next_u64());
        }
        check_sum6(X);
        for (auto &x : X) {
            int64_t e = (int64_t)e0 + (int64_t)(next_u64() % 3) - 1;
            e = e < 0 ? 0 : (e > 2047 ? 2047 : e);
            const uint64_t f = (next_u64() & 1) ? next_u64() : next_u64() & ~((1ull << (next_u64() % 53)) - 1);
            x = make(sg, (uint64_t)e, f);
        }
        check_sum6(X);
        const uint64_t e1 = 1 + next_u64() % 2040;
        for (auto &x : X) x = make(sg, e1 + next_u64() % 9, (next_u64() & 1) ? kFrac : (next_u64() & 0xFFF0000000000ull));
        check_sum6(X);
        const uint64_t t = make(sg, 2030 + next_u64() % 18, kFrac - next_u64() % 8);
        for (auto &x : X) x = t;
        check_sum6(X);
        for (auto &x : X) x = bits((double)(next_u64() >> 11) * 0x1p-53);
        check_sum6(X);
        for (auto &x : X) {
            const uint64_t r = next_u64() % 4;
            x = r == 0 ? make(sg, 0, 0) : r == 1 ? make(sg, 0, next_u64()) : make(sg, next_u64() % 12, next_u64());
        }
        check_sum6(X);
    }
    // six-operand sums with a zero tolerated in the first or second slot
    zero_slot_cases<0>(n / 2);
    zero_slot_cases<1>(n / 2);
    std::printf("mismatches %llu cases %llu sum4_taken %llu sum6_taken %llu sum6z_taken %llu sum4z_taken %llu\n",
                (unsigned long long)mismatches, (unsigned long long)cases, (unsigned long long)sum4_taken,
                (unsigned long long)sum6_taken, (unsigned long long)sum6z_taken, (unsigned long long)sum4z_taken);
    return mismatches != 0;
}
