// situ_device.cuh — device-side helpers shared by the SiTU-GLU kernels: vector types, streaming
// loads and stores (inline PTX), bf16 and FP8 (E4M3) conversions, warp reductions.
#pragma once

#include <stdint.h>

namespace situ {

// NW consecutive 32-bit words (2·NW bf16): NW = 4 is a 16-byte chunk, NW = 8 a 32-byte chunk.
template <int NW>
struct Vec {
    uint32_t w[NW];
};

// Streaming load. NC = true reads through the non-coherent path (inputs no thread writes);
// NC = false through the coherent path (x, which dx may alias in place). NOALLOC adds the
// L1::no_allocate hint (measured faster for the 32-byte backward, slower for the 16-byte one).
template <int NW, bool NC, bool NOALLOC = true>
__device__ __forceinline__ Vec<NW> ld_stream(const Vec<NW>* p) {
    Vec<NW> v;
    if constexpr (NW == 4) {
        if constexpr (NC && NOALLOC)
            asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
                : "l"(p));
        else if constexpr (NC)
            asm("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
                : "l"(p));
        else if constexpr (NOALLOC)
            asm("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
                : "l"(p));
        else
            asm("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];"
                : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
                : "l"(p));
    } else {
        static_assert(NW == 8, "16- or 32-byte vectors");
        static_assert(NOALLOC, "the 32-byte path always uses L1::no_allocate");
        if constexpr (NC)
            asm("ld.global.nc.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]), "=r"(v.w[4]), "=r"(v.w[5]),
                  "=r"(v.w[6]), "=r"(v.w[7])
                : "l"(p));
        else
            asm("ld.global.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]), "=r"(v.w[4]), "=r"(v.w[5]),
                  "=r"(v.w[6]), "=r"(v.w[7])
                : "l"(p));
    }
    return v;
}

// Streaming (evict-first) store.
template <int NW>
__device__ __forceinline__ void st_stream(Vec<NW>* p, const Vec<NW>& v) {
    if constexpr (NW == 4) {
        asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]),
                     "r"(v.w[3])
                     : "memory");
    } else {
        asm volatile("st.global.cs.v8.u32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(v.w[0]), "r"(v.w[1]),
                     "r"(v.w[2]), "r"(v.w[3]), "r"(v.w[4]), "r"(v.w[5]), "r"(v.w[6]), "r"(v.w[7])
                     : "memory");
    }
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

// Two fp32 -> packed bf16x2 (round to nearest even); lo goes to the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint16_t f32_to_bf16(float f) { return (uint16_t)(pack_bf16x2(f, 0.0f) & 0xFFFFu); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}


// FP8 E4M3 (OCP): two fp32 -> two codes, round to nearest even, finite values saturated to
// +-448 (cvt.rn.satfinite.e4m3x2.f32); lo goes to the low byte.
__device__ __forceinline__ uint16_t e4m3x2_from_f32(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two E4M3 codes (low byte, high byte) -> their exact values as fp32 (through f16, which
// holds every E4M3 value exactly).
__device__ __forceinline__ void e4m3x2_to_f32(uint16_t codes, float& lo, float& hi) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(codes));
    uint16_t l16 = (uint16_t)(h2 & 0xFFFFu), h16 = (uint16_t)(h2 >> 16);
    asm("cvt.f32.f16 %0, %1;" : "=f"(lo) : "h"(l16));
    asm("cvt.f32.f16 %0, %1;" : "=f"(hi) : "h"(h16));
}

// Max over the 16 lanes of a half-warp (lanes 0-15 or 16-31).
__device__ __forceinline__ float halfwarp_max(float v) {
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

}  // namespace situ
