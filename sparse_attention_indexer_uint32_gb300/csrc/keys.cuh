// keys.cuh -- the order-preserving fp32 -> uint32 key map and its inverse,
// used by every select kernel and by the stand-alone key-map entry point.
#pragma once

#include <cstdint>

namespace topkidx {

// Order-preserving fp32 -> uint32 map (DistRadixTopK README "Ultra Low
// Latency Distributed Radix TopK Indexer Via NoC", "Distributed Radix Sort
// via NoC", second point: a bin map under which a larger bin means a larger
// score).  -0.0 is first folded onto +0.0 so the two tie; then the sign bit
// is flipped for non-negative values and every bit is flipped for negative
// ones, which makes unsigned key order equal to IEEE order.  NaNs keep their
// bits: positive NaNs land above +inf (a larger payload higher), negative
// NaNs below -inf (a larger payload lower).
__device__ __forceinline__ uint32_t score_key(float x) {
    uint32_t u = __float_as_uint(x);
    u = (u == 0x80000000u) ? 0u : u;
    const uint32_t m = static_cast<uint32_t>(static_cast<int32_t>(u) >> 31) | 0x80000000u;
    return u ^ m;
}

// The float whose key is `key` (the inverse of score_key on keys of non-NaN
// floats): score_key(x) >= key <=> !(x < key_float(key)) for every non-NaN
// x.  key == 0 gives a NaN, so that the compare lets every element through;
// NaN elements always pass the compare and are sorted out by their exact key.
__device__ __forceinline__ float key_float(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

}  // namespace topkidx
