// ct_gen_io.cuh -- loads and stores of the general kernels for any
// alignment: 8 bf16 (or 16 bytes) shifted out of the two aligned 16-byte
// blocks that cover them, and 8- / 16-byte stores as one vector store when
// aligned, else as aligned 4-byte words shifted across registers plus a 1- to
// 3-byte head and tail (byte by byte when cut short).  Shared by the general
// kernels and by the direct-load kernel's transposed stores when rows is not a
// multiple of 16.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace ct {
namespace gen {

// Word k + j of w[0..7], k in 0..3 (static indexing only).
__device__ __forceinline__ uint32_t pick(const uint32_t (&w)[8], int j, int k) {
    const uint32_t a = w[j], b = w[j + 1], c = w[j + 2], d = w[j + 3];
    return k == 0 ? a : k == 1 ? b : k == 2 ? c : d;
}

// The 8 bf16 that start at element m (0..7) of the 16 held by lo, hi.
__device__ __forceinline__ uint4 extract8(const uint4& lo, const uint4& hi, int m) {
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    const int k = m >> 1;
    const uint32_t t0 = pick(w, 0, k), t1 = pick(w, 1, k), t2 = pick(w, 2, k),
                   t3 = pick(w, 3, k), t4 = pick(w, 4, k);
    if ((m & 1) == 0) return make_uint4(t0, t1, t2, t3);
    // odd start: the high half of word k + j, then the low half of word k + j + 1
    return make_uint4(__byte_perm(t0, t1, 0x5432), __byte_perm(t1, t2, 0x5432),
                      __byte_perm(t2, t3, 0x5432), __byte_perm(t3, t4, 0x5432));
}

// Zero the elements n..7 of an 8-element chunk.
__device__ __forceinline__ uint4 keep_first(uint4 v, int n) {
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 8; ++i)
        if (i >= n) w[i >> 1] &= (i & 1) ? 0x0000FFFFu : 0xFFFF0000u;
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// The 16 bytes that start at byte m (0..15) of the 32 held by lo, hi.
__device__ __forceinline__ uint4 extract16(const uint4& lo, const uint4& hi, int m) {
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    const int k = m >> 2, sh = 8 * (m & 3);
    const uint32_t t0 = pick(w, 0, k), t1 = pick(w, 1, k), t2 = pick(w, 2, k),
                   t3 = pick(w, 3, k), t4 = pick(w, 4, k);
    return make_uint4(__funnelshift_r(t0, t1, sh), __funnelshift_r(t1, t2, sh),
                      __funnelshift_r(t2, t3, sh), __funnelshift_r(t3, t4, sh));
}

// Zero the bytes n..15.
__device__ __forceinline__ uint4 keep_first_bytes(uint4 v, int n) {
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 16; ++i)
        if (i >= n) w[i >> 2] &= ~(0xFFu << (8 * (i & 3)));
    return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ uint8_t byte_of(const uint32_t (&w)[4], int i) {
    return static_cast<uint8_t>(w[i >> 2] >> (8 * (i & 3)));
}

// Store the K words d[0..K-1] (4K bytes) at dst, where h = dst & 3 is 1, 2
// or 3: the 4 - h head bytes, K - 1 whole aligned words shifted across
// registers (funnel shift by 8h bits), then the h tail bytes.
template <int K>
__device__ __forceinline__ void store_words_unaligned(uint8_t* dst, const uint32_t (&d)[K], int h) {
    const uint32_t first = d[0], last = d[K - 1];
    uint8_t* base = dst - h;   // 4-byte aligned
#pragma unroll
    for (int j = 1; j < K; ++j)
        reinterpret_cast<uint32_t*>(base)[j] = __funnelshift_r(d[j - 1], d[j], 8 * (4 - h));
    uint8_t* tail = base + 4 * K;
    if (h == 1) {
        dst[0] = static_cast<uint8_t>(first);
        *reinterpret_cast<uint16_t*>(dst + 1) = static_cast<uint16_t>(first >> 8);
        tail[0] = static_cast<uint8_t>(last >> 24);
    } else if (h == 2) {
        *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(first);
        *reinterpret_cast<uint16_t*>(tail) = static_cast<uint16_t>(last >> 16);
    } else {
        dst[0] = static_cast<uint8_t>(first);
        *reinterpret_cast<uint16_t*>(tail) = static_cast<uint16_t>(last >> 8);
        tail[2] = static_cast<uint8_t>(last >> 24);
    }
}

// Bytes 0..n-1 of the 16 in w to dst.
__device__ __forceinline__ void store16(uint8_t* dst, const uint32_t (&w)[4], int n) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(dst);
    if (n == 16) {
        if ((a & 15) == 0) {
            __stcs(reinterpret_cast<uint4*>(dst), make_uint4(w[0], w[1], w[2], w[3]));
            return;
        }
        if ((a & 7) == 0) {
            __stcs(reinterpret_cast<uint2*>(dst), make_uint2(w[0], w[1]));
            __stcs(reinterpret_cast<uint2*>(dst + 8), make_uint2(w[2], w[3]));
            return;
        }
        if ((a & 3) == 0) {
#pragma unroll
            for (int j = 0; j < 4; ++j) reinterpret_cast<uint32_t*>(dst)[j] = w[j];
            return;
        }
        store_words_unaligned<4>(dst, w, static_cast<int>(a & 3));
        return;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i)
        if (i < n) dst[i] = byte_of(w, i);
}

// Bytes 0..n-1 of the 8 in q to dst.
__device__ __forceinline__ void store8(uint8_t* dst, uint2 q, int n) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(dst);
    if (n == 8) {
        if ((a & 7) == 0) {
            __stcs(reinterpret_cast<uint2*>(dst), q);
            return;
        }
        if ((a & 3) == 0) {
            reinterpret_cast<uint32_t*>(dst)[0] = q.x;
            reinterpret_cast<uint32_t*>(dst)[1] = q.y;
            return;
        }
        const uint32_t d[2] = {q.x, q.y};
        store_words_unaligned<2>(dst, d, static_cast<int>(a & 3));
        return;
    }
    const uint32_t w[4] = {q.x, q.y, 0u, 0u};
#pragma unroll
    for (int i = 0; i < 8; ++i)
        if (i < n) dst[i] = byte_of(w, i);
}

}  // namespace gen

}  // namespace ct
