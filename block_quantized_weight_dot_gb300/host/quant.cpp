// quant.cpp -- float weights -> canonical Q4_0 / Q8_0 / INT8-B64 blocks on the
// host, the load-time step before lean_pack ("oxinfer" crate page, How it
// works: quant.rs quantizes weights into Q8 and Q4_0 blocks at load time;
// "wgpu-llm" README, INT8 mode: a quantizer with block size 64).
//
// The pages give no rounding rule; the one taken (include/lean_quant.h):
//   Q8_0 / INT8-B64: d = binary16 nearest to max|w| / 127 (ties to even),
//                    q = nearest integer to w / d (ties away from zero) in
//                    [-127, 127];
//   Q4_0:            m = the first element of largest |w|, d = binary16
//                    nearest to m / -8, q = nearest integer to w / d (ties
//                    away from zero) + 8 in [0, 15];
//   a scale that rounds to zero is stored as +0 with every value 0.
// The quotients are taken in double, where w / d is correctly rounded and
// cannot land on or leave a half-way point, so the codes are those of the
// exact quotients; |w / d| stays below 2 * 127 (the scale is at least half
// of max|w| / 127 or |m| / 8 once rounded), far inside the integer
// conversion used to round.  Host code only: no kernel depends on this file.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

#include "../../include/lean_quant.h"

namespace {

// binary16 bits of the value nearest to v (ties to even), from the bits of
// the double: keep the significand down to the binary16 quantum of v's
// binade (2^-24 below 2^-14), rounding the dropped bits.  False if v is not
// finite or rounds past 65504.
bool half_bits(double v, uint16_t &out) {
    if (!std::isfinite(v)) return false;
    uint64_t b;
    std::memcpy(&b, &v, sizeof b);
    const uint16_t sign = (uint16_t)((b >> 48) & 0x8000u);
    const int raw = (int)((b >> 52) & 0x7ff);
    if (raw == 0) {  // zero or a double subnormal: far below 2^-25
        out = sign;
        return true;
    }
    const int e = raw - 1023;                                   // v in [2^e, 2^(e+1))
    const uint64_t mant = (b & ((1ull << 52) - 1)) | (1ull << 52);  // v = mant * 2^(e-52)
    if (e > 15) return false;
    const int quantum = (e < -14 ? -14 : e) - 10;               // binary16 spacing 2^quantum
    const int shift = quantum - (e - 52);                       // >= 42
    uint64_t k = 0;
    if (shift < 64) {
        k = mant >> shift;
        const uint64_t rest = mant & ((1ull << shift) - 1), half = 1ull << (shift - 1);
        if (rest > half || (rest == half && (k & 1))) ++k;
    }
    // subnormal: k * 2^-24 with k <= 1024 (1024 is the smallest normal, same
    // bits); normal: exponent field e + 15 and k in [1024, 2048], where 2048
    // carries into the exponent
    const uint32_t h = e < -14 ? (uint32_t)k : (uint32_t)(((e + 15) << 10) + (int)(k - 1024));
    if (h >= 0x7c00u) return false;
    out = (uint16_t)(h | sign);
    return true;
}

// nearest integer to t, ties away from zero, for |t| < 2^31: the conversion
// truncates toward zero, and t - trunc(t) is exact
inline double round_away(double t) {
    const double r = (double)(int64_t)t;
    const double f = t - r;
    return f >= 0.5 ? r + 1.0 : (f <= -0.5 ? r - 1.0 : r);
}

double half_value(uint16_t h) {
    const int e = (h >> 10) & 0x1f, f = h & 0x3ff;
    const double a = e == 0 ? std::ldexp((double)f, -24) : std::ldexp((double)(f + 1024), e - 25);
    return (h & 0x8000) ? -a : a;
}

int block_elems_of(int fmt) {
    return fmt == LEAN_Q4_0 ? 32 : fmt == LEAN_Q8_0 ? 32 : fmt == LEAN_I8_B64 ? 64 : 0;
}

// One block of `be` weights into `blk` (canonical layout).  False on a
// non-finite weight or a scale past the binary16 range.
bool quantize_block(int fmt, const float *w, uint8_t *blk) {
    const int be = block_elems_of(fmt);
    for (int j = 0; j < be; ++j)
        if (!std::isfinite(w[j])) return false;
    double pick = 0.0;  // Q4_0: the first element of largest magnitude; else max |w|
    for (int j = 0; j < be; ++j) {
        const double a = std::fabs((double)w[j]);
        if (a > std::fabs(pick)) pick = fmt == LEAN_Q4_0 ? (double)w[j] : a;
    }
    uint16_t db = 0;
    if (pick != 0.0 && !half_bits(fmt == LEAN_Q4_0 ? pick / -8.0 : pick / 127.0, db)) return false;
    if ((db & 0x7fffu) == 0) db = 0;
    const double d = half_value(db);
    blk[0] = (uint8_t)(db & 0xff);
    blk[1] = (uint8_t)(db >> 8);
    if (fmt == LEAN_Q4_0) {
        uint8_t q[32];
        for (int j = 0; j < 32; ++j) {
            double t = d == 0.0 ? 8.0 : round_away((double)w[j] / d) + 8.0;
            t = t < 0.0 ? 0.0 : t > 15.0 ? 15.0 : t;
            q[j] = (uint8_t)t;
        }
        for (int j = 0; j < 16; ++j) blk[2 + j] = (uint8_t)(q[j] | (q[j + 16] << 4));
    } else {
        for (int j = 0; j < be; ++j) {
            double t = d == 0.0 ? 0.0 : round_away((double)w[j] / d);
            t = t < -127.0 ? -127.0 : t > 127.0 ? 127.0 : t;
            blk[2 + j] = (uint8_t)(int8_t)(int)t;
        }
    }
    return true;
}

}  // namespace

extern "C" {

lean_status lean_quantize(int fmt, const float *w_host, void *canon_host, int64_t N, int64_t K,
                          int threads) {
    const int be = block_elems_of(fmt);
    if (be == 0) return LEAN_ERR_FORMAT;
    if (!w_host || !canon_host) return LEAN_ERR_NULL;
    if (N <= 0 || K <= 0 || K % be != 0 || threads < 0) return LEAN_ERR_SHAPE;
    const int64_t nb = K / be, bb = be == 32 ? (fmt == LEAN_Q4_0 ? 18 : 34) : 66;
    uint8_t *out = static_cast<uint8_t *>(canon_host);
    int nt = threads > 0 ? threads : (int)std::thread::hardware_concurrency();
    if (nt < 1) nt = 1;
    if ((int64_t)nt > N) nt = (int)N;
    std::atomic<bool> ok{true};
    auto rows = [&](int64_t r0, int64_t r1) {
        for (int64_t n = r0; n < r1 && ok.load(std::memory_order_relaxed); ++n)
            for (int64_t b = 0; b < nb; ++b)
                if (!quantize_block(fmt, w_host + n * K + b * be, out + (n * nb + b) * bb)) {
                    ok.store(false);
                    return;
                }
    };
    if (nt == 1) {
        rows(0, N);
    } else {
        std::vector<std::thread> pool;
        for (int t = 0; t < nt; ++t) pool.emplace_back(rows, N * t / nt, N * (t + 1) / nt);
        for (auto &th : pool) th.join();
    }
    return ok.load() ? LEAN_OK : LEAN_ERR_SHAPE;
}

}  // extern "C"
