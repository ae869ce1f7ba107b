// Coreset target in integer arithmetic: ceil(top_p * total) where the product
// is taken the IEEE way, fp32 top_p times total rounded to double, the product
// rounded to nearest-even double (the rounding of a double multiply), and the
// ceiling of that value, clamped to [1, total].  Written with integers (a
// 24 x 53-bit product in 128 bits) so it needs no fp64 unit; compiles as
// plain C++ too (the host test checks it against double arithmetic).
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define MOESTEP_HD __host__ __device__ __forceinline__
#else
#define MOESTEP_HD inline
#endif

namespace moestep {

MOESTEP_HD int clz_u64(unsigned long long v) {
#if defined(__CUDA_ARCH__)
    return __clzll(static_cast<long long>(v));
#else
    return v ? __builtin_clzll(v) : 64;
#endif
}

MOESTEP_HD int bit_length_u128(unsigned __int128 v) {
    const unsigned long long hi = static_cast<unsigned long long>(v >> 64);
    const unsigned long long lo = static_cast<unsigned long long>(v);
    return hi ? 128 - clz_u64(hi) : 64 - clz_u64(lo);
}

// v rounded to `keep` significant bits, nearest-even: returns the mantissa and
// adds the dropped bit count to *shift.
MOESTEP_HD unsigned __int128 round_bits_rne(unsigned __int128 v, int keep, int* shift) {
    const int bits = bit_length_u128(v);
    if (bits <= keep) return v;
    int sh = bits - keep;
    unsigned __int128 q = v >> sh;
    const unsigned __int128 rem = v & ((static_cast<unsigned __int128>(1) << sh) - 1);
    const unsigned __int128 half = static_cast<unsigned __int128>(1) << (sh - 1);
    if (rem > half || (rem == half && (q & 1))) ++q;
    if (q >> keep) {  // carried into a new bit
        q >>= 1;
        ++sh;
    }
    *shift += sh;
    return q;
}

// ceil(RN(top_p * RN(total))) clamped to [1, total]; 0 < top_p < 1, total > 0.
MOESTEP_HD long long coreset_target(float top_p, long long total) {
    // total as a double: mantissa md (<= 53 bits) times 2^ed
    int ed = 0;
    const unsigned __int128 md = round_bits_rne(static_cast<unsigned __int128>(total), 53, &ed);
    // top_p = mt * 2^et exactly
    uint32_t b;
#if defined(__CUDA_ARCH__)
    b = __float_as_uint(top_p);
#else
    __builtin_memcpy(&b, &top_p, 4);
#endif
    const int ex = static_cast<int>((b >> 23) & 0xffu);
    const unsigned long long mt = (b & 0x7fffffu) | (ex ? 0x800000u : 0u);
    const int et = (ex ? ex : 1) - 150;
    // the product, rounded to 53 bits
    int e = et + ed;
    const unsigned __int128 p = round_bits_rne(static_cast<unsigned __int128>(mt) * md, 53, &e);
    unsigned __int128 v;  // ceil(p * 2^e)
    if (p == 0) {
        v = 0;
    } else if (e >= 0) {
        v = e >= 64 ? static_cast<unsigned __int128>(total) : p << e;
    } else if (-e >= 128) {
        v = 1;
    } else {
        const int sh = -e;
        const bool frac = (p & ((static_cast<unsigned __int128>(1) << sh) - 1)) != 0;
        v = (p >> sh) + (frac ? 1 : 0);
    }
    long long target = v > static_cast<unsigned __int128>(total) ? total : static_cast<long long>(v);
    if (target < 1) target = 1;
    if (target > total) target = total;
    return target;
}

}  // namespace moestep
