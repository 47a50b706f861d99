// Register-fragment helpers shared by the warp-streaming expand and the fused
// shrink+expand kernels (mma.sync m16n8k16, fp32 accumulate).
//
// Contraction-index permutation used for expand: in one 16-wide k step a
// thread's A / B slots {2q, 2q+1, 2q+8, 2q+9} hold the ranks 4q .. 4q+3, so
// the thread reads 4 consecutive ranks (8 bytes of a B row, 16 bytes of y).
// Output-column permutation: n-tile i, column c -> 8*(c/2) + 2i + c%2, so a
// thread's accumulators are 8 consecutive output columns.
#pragma once

#include "common.cuh"

namespace lora {

template <typename E> struct Pack;
template <> struct Pack<__half> {
    static __device__ __forceinline__ uint32_t pack(float a, float b) {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    static __device__ __forceinline__ float2 unpack(uint32_t w) {
        return __half22float2(*reinterpret_cast<__half2 *>(&w));
    }
};
template <> struct Pack<__nv_bfloat16> {
    static __device__ __forceinline__ uint32_t pack(float a, float b) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    static __device__ __forceinline__ float2 unpack(uint32_t w) {
        return __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&w));
    }
};

// Eight floats <-> eight fp16/bf16 values in one 16-byte word (round to nearest even).
template <typename E>
__device__ __forceinline__ uint4 pack8(const float (&v)[8]) {
    uint4 r;
    uint32_t *w = reinterpret_cast<uint32_t *>(&r);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        E lo = Elem<E>::from_f(v[2 * k]), hi = Elem<E>::from_f(v[2 * k + 1]);
        w[k] = (uint32_t)(*reinterpret_cast<uint16_t *>(&lo)) |
               ((uint32_t)(*reinterpret_cast<uint16_t *>(&hi)) << 16);
    }
    return r;
}

template <typename E>
__device__ __forceinline__ void unpack8(uint4 r, float (&v)[8]) {
    const uint32_t *w = reinterpret_cast<const uint32_t *>(&r);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        uint16_t lo = (uint16_t)(w[k] & 0xffffu), hi = (uint16_t)(w[k] >> 16);
        v[2 * k] = Elem<E>::to_f(*reinterpret_cast<E *>(&lo));
        v[2 * k + 1] = Elem<E>::to_f(*reinterpret_cast<E *>(&hi));
    }
}

// v = hi + lo with hi = round(v) and lo = round(v - hi) in the weight type.
template <typename E>
__device__ __forceinline__ void split_hilo8(const float (&v)[8], uint4 &hi, uint4 &lo) {
    float h[8], l[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        h[k] = Elem<E>::to_f(Elem<E>::from_f(v[k]));
        l[k] = v[k] - h[k];
    }
    hi = pack8<E>(h);
    lo = pack8<E>(l);
}

// Power-of-two factor 2^k as a float, k in [-126, 127].
__device__ __forceinline__ float exp2i(int k) { return __int_as_float((127 + k) << 23); }

// Per-row exponent e with max|y_row| * 2^-e < 1 (frexp-style), clamped.
__device__ __forceinline__ int row_exponent(float m) {
    const int be = (__float_as_int(m) >> 23) & 0xff;
    return min(max(be - 126, -125), 126);
}

// B fragments of one 32-column block: n-tile i, k step ks -> 4 ranks of row
// n = c0 + 8*(g/2) + 2i + g%2 of Bl (an [Ns, R] matrix), ranks >= rl zeroed.
template <typename E, int KSMAX>
__device__ __forceinline__ void load_bfrags(uint2 (&bf)[KSMAX][4], const E *Bl, int Ns, int R,
                                            int c0, int rl, int KS, int g, int q) {
#pragma unroll
    for (int ks = 0; ks < KSMAX; ++ks)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            bf[ks][i] = make_uint2(0, 0);
            const int n = c0 + 8 * (g >> 1) + 2 * i + (g & 1);
            const int k = ks * 16 + 4 * q;
            if (ks < KS && n < Ns && k < rl) {
                uint2 v = __ldg(reinterpret_cast<const uint2 *>(Bl + (int64_t)n * R + k));
                const int nv = rl - k;  // valid ranks among these 4
                if (nv < 4) {
                    v.y = nv <= 2 ? 0u : (v.y & 0xffffu);
                    if (nv < 2) v.x &= 0xffffu;
                }
                bf[ks][i] = v;
            }
        }
}

// y fragments (hi + lo pair of the weight type) of MB m16 blocks for ranks
// [0, rl) of the y rows `rows` (y row pointer = yb + row * ldy), each row
// scaled by a power of two; fscale receives scale * 2^e per row.
// COHERENT: y was written earlier in the same kernel (L2 loads, not the
// read-only path).
template <typename E, int MB, int KSMAX, bool COHERENT>
__device__ __forceinline__ void build_yfrags(uint32_t (&ah)[MB][KSMAX][4],
                                             uint32_t (&al)[MB][KSMAX][4], float (&fscale)[MB][2],
                                             const int (&rows)[MB][2], const float *yb, int64_t ldy,
                                             int rl, int KS, float scale, bool y_vec, int q) {
    float yv[MB][2][KSMAX][4];
#pragma unroll
    for (int mm = 0; mm < MB; ++mm)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int row = rows[mm][h];
            const float *yr = yb + (int64_t)(row < 0 ? 0 : row) * ldy;
#pragma unroll
            for (int ks = 0; ks < KSMAX; ++ks) {
                const int k = ks * 16 + 4 * q;
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (row >= 0 && ks < KS && k < rl) {
                    if (y_vec && k + 4 <= rl) {
                        v = COHERENT ? __ldcg(reinterpret_cast<const float4 *>(yr + k))
                                     : __ldg(reinterpret_cast<const float4 *>(yr + k));
                    } else {
                        v.x = COHERENT ? __ldcg(yr + k) : __ldg(yr + k);
                        if (k + 1 < rl) v.y = COHERENT ? __ldcg(yr + k + 1) : __ldg(yr + k + 1);
                        if (k + 2 < rl) v.z = COHERENT ? __ldcg(yr + k + 2) : __ldg(yr + k + 2);
                        if (k + 3 < rl) v.w = COHERENT ? __ldcg(yr + k + 3) : __ldg(yr + k + 3);
                    }
                }
                yv[mm][h][ks][0] = v.x;
                yv[mm][h][ks][1] = v.y;
                yv[mm][h][ks][2] = v.z;
                yv[mm][h][ks][3] = v.w;
            }
        }
#pragma unroll
    for (int mm = 0; mm < MB; ++mm)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float mx = 0.f;
#pragma unroll
            for (int ks = 0; ks < KSMAX; ++ks)
#pragma unroll
                for (int j = 0; j < 4; ++j) mx = fmaxf(mx, fabsf(yv[mm][h][ks][j]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const int e = row_exponent(mx);
            fscale[mm][h] = scale * exp2i(e);
            const float inv = exp2i(-e);
#pragma unroll
            for (int ks = 0; ks < KSMAX; ++ks)
#pragma unroll
                for (int j = 0; j < 4; ++j) yv[mm][h][ks][j] *= inv;
        }
#pragma unroll
    for (int mm = 0; mm < MB; ++mm)
#pragma unroll
        for (int ks = 0; ks < KSMAX; ++ks)
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                // a0: (row g, ranks 4q, 4q+1)  a1: (row g+8, 4q, 4q+1)
                // a2: (row g, 4q+2, 4q+3)     a3: (row g+8, 4q+2, 4q+3)
                const int h = r & 1, j = (r >> 1) * 2;
                const float v0 = yv[mm][h][ks][j], v1 = yv[mm][h][ks][j + 1];
                const uint32_t hw = Pack<E>::pack(v0, v1);
                const float2 hf = Pack<E>::unpack(hw);
                ah[mm][ks][r] = hw;
                al[mm][ks][r] = Pack<E>::pack(v0 - hf.x, v1 - hf.y);
            }
}

// One m16 block of a 32-column expand unit: MMAs over KS k steps, then the
// epilogue out = (add ? out_old : 0) + fscale_row * acc, stored with 16-byte
// stores at column `col` of rows `rows[h]`.
template <typename E, bool ADD, int KSMAX>
__device__ __forceinline__ void expand_block(E *out, int64_t ldo, int64_t col, const int (&rows)[2],
                                             const uint32_t (&ah)[KSMAX][4],
                                             const uint32_t (&al)[KSMAX][4],
                                             const uint2 (&bf)[KSMAX][4], const float (&fs)[2],
                                             const uint4 (&old)[2], int KS, bool col_ok) {
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[i][k] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KSMAX; ++ks) {
        if (ks < KS) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                mma16816<E>(acc[i], ah[ks], bf[ks][i].x, bf[ks][i].y);
                mma16816<E>(acc[i], al[ks], bf[ks][i].x, bf[ks][i].y);
            }
        }
    }
    if (!col_ok) return;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int row = rows[h];
        if (row < 0) continue;
        const float f = fs[h];
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float r0 = f * acc[k][2 * h], r1 = f * acc[k][2 * h + 1];
            if (ADD) {
                const float2 o = Pack<E>::unpack(reinterpret_cast<const uint32_t *>(&old[h])[k]);
                r0 = fmaf(f, acc[k][2 * h], o.x);
                r1 = fmaf(f, acc[k][2 * h + 1], o.y);
            }
            w[k] = Pack<E>::pack(r0, r1);
        }
        st_global_v4(out + (int64_t)row * ldo + col, make_uint4(w[0], w[1], w[2], w[3]));
    }
}

}  // namespace lora
