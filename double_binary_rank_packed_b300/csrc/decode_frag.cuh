// Register-fragment helpers shared by the decode kernels (mma.sync m16n8k16
// with fp16 operands and fp32 accumulators; activation operands in the perm8
// K order, sign operands unpacked with sign_pairs8).
#pragma once

#include "common.cuh"

namespace dbfk {

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Two m16n8k16 MMAs (k 0..15 and 16..31 of one packed word) for rows g and
// g+8 of a 16-row block: pa / pv are the sign pairs of the two rows, b the
// lane's four activation pairs (see perm8_pos and sign_pairs8).
__device__ __forceinline__ void mma_word8(float (&acc)[4], const uint32_t (&pa)[4], const uint32_t (&pv)[4],
                                          const uint32_t (&b)[4]) {
    mma_16816(acc, pa[0], pv[0], pa[1], pv[1], b[0], b[1]);
    mma_16816(acc, pa[2], pv[2], pa[3], pv[3], b[2], b[3]);
}

// The ragged or unaligned case of load_x8, kept out of line: it is rare, and
// inlined at every unrolled call site it would multiply the kernels' code.
static __device__ __noinline__ uint4 load_x8_slow(const __nv_bfloat16 *row, int k0, int kmax) {
    const uint16_t *r16 = reinterpret_cast<const uint16_t *>(row);
    uint16_t v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = (k0 + j < kmax) ? r16[k0 + j] : uint16_t(0);
    return make_uint4(v[0] | (uint32_t(v[1]) << 16), v[2] | (uint32_t(v[3]) << 16), v[4] | (uint32_t(v[5]) << 16),
                      v[6] | (uint32_t(v[7]) << 16));
}

// 8 bf16 of x (k0 .. k0+7 of one row, zero at k >= kmax) with plain
// coherent loads: x is written by an earlier kernel.
__device__ __forceinline__ uint4 load_x8(const __nv_bfloat16 *row, int k0, int kmax, bool vec) {
    if (vec && k0 + 8 <= kmax) return *reinterpret_cast<const uint4 *>(row + k0);
    return load_x8_slow(row, k0, kmax);
}

// The lane's four B pairs of one word from 8 bf16 x (physical k 8c..8c+7)
// and the matching 8 fp16 gamma: pair j = fp16(gamma*x) at (8c+j, 8c+j+4).
__device__ __forceinline__ void x_pairs(const uint4 &xv, const uint4 &gv, uint32_t (&b)[4]) {
    const float2 g01 = __half22float2(*reinterpret_cast<const __half2 *>(&gv.x));
    const float2 g23 = __half22float2(*reinterpret_cast<const __half2 *>(&gv.y));
    const float2 g45 = __half22float2(*reinterpret_cast<const __half2 *>(&gv.z));
    const float2 g67 = __half22float2(*reinterpret_cast<const __half2 *>(&gv.w));
    __half2 h;
    h = __floats2half2_rn(bf16lo(xv.x) * g01.x, bf16lo(xv.z) * g45.x);
    b[0] = *reinterpret_cast<uint32_t *>(&h);
    h = __floats2half2_rn(bf16hi(xv.x) * g01.y, bf16hi(xv.z) * g45.y);
    b[1] = *reinterpret_cast<uint32_t *>(&h);
    h = __floats2half2_rn(bf16lo(xv.y) * g23.x, bf16lo(xv.w) * g67.x);
    b[2] = *reinterpret_cast<uint32_t *>(&h);
    h = __floats2half2_rn(bf16hi(xv.y) * g23.y, bf16hi(xv.w) * g67.y);
    b[3] = *reinterpret_cast<uint32_t *>(&h);
}

template <int CT>
__device__ __forceinline__ void zero_acc(float (&acc)[CT][4]) {
#pragma unroll
    for (int ct = 0; ct < CT; ++ct) acc[ct][0] = acc[ct][1] = acc[ct][2] = acc[ct][3] = 0.f;
}

// Fragment (16 rows x 8*CT columns) -> 32-bit shared-memory address `base`
// (row stride ld floats) of the CTA `rank` of the cluster (or of this CTA when
// remote is false).
template <int CT>
__device__ __forceinline__ void put_frag(uint32_t base, int ld, const float (&acc)[CT][4], int lane, bool remote,
                                         uint32_t rank) {
    const int g = lane >> 2, c = lane & 3;
#pragma unroll
    for (int ct = 0; ct < CT; ++ct) {
        const uint32_t a0 = base + 4u * static_cast<uint32_t>(g * ld + ct * 8 + 2 * c);
        const uint32_t a1 = a0 + 4u * static_cast<uint32_t>(8 * ld);
        if (remote) {
            asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(mapa_shared(a0, rank)), "f"(acc[ct][0]),
                         "f"(acc[ct][1])
                         : "memory");
            asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(mapa_shared(a1, rank)), "f"(acc[ct][2]),
                         "f"(acc[ct][3])
                         : "memory");
        } else {
            asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(a0), "f"(acc[ct][0]), "f"(acc[ct][1]) : "memory");
            asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(a1), "f"(acc[ct][2]), "f"(acc[ct][3]) : "memory");
        }
    }
}

__device__ __forceinline__ void add4(float4 &u, const float4 &o) {
    u.x += o.x;
    u.y += o.y;
    u.z += o.z;
    u.w += o.w;
}

}  // namespace dbfk
