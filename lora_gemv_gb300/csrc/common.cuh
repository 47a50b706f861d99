// Device helpers shared by the plan, shrink and expand kernels (sm_103a).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <limits.h>
#include <stdint.h>

#include "lora_gemv.h"

namespace lora {

constexpr int kTile = LORA_TILE_TOKENS;  // tokens per plan tile
constexpr int kMaxSlices = LORA_MAX_SLICES;

// ------------------------------------------------------------------ plan view
struct PlanView {
    int32_t *hdr;          // LORA_HDR_WORDS header words (kernels may OR error bits)
    const int32_t *perm;   // [T]
    const int4 *tiles;     // [max_tiles] {lora, p0, n, group}
};

__device__ __forceinline__ bool plan_matches(const PlanView &p, int T, int L) {
    const volatile int32_t *h = p.hdr;
    return h[LORA_HDR_MAGIC] == LORA_PLAN_MAGIC && h[LORA_HDR_T] == T && h[LORA_HDR_L] == L;
}

// ------------------------------------------------------------------ dtype traits
template <typename E> struct Elem;
template <> struct Elem<__half> {
    static __device__ __forceinline__ float to_f(__half v) { return __half2float(v); }
    static __device__ __forceinline__ __half from_f(float v) { return __float2half_rn(v); }
};
template <> struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
    static __device__ __forceinline__ __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};

// mma.sync m16n8k16, fp32 accumulate; A row-major (4 regs), B col-major (2 regs).
template <typename E>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1);
template <>
__device__ __forceinline__ void mma16816<__half>(float (&d)[4], const uint32_t (&a)[4],
                                                 uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
template <>
__device__ __forceinline__ void mma16816<__nv_bfloat16>(float (&d)[4], const uint32_t (&a)[4],
                                                        uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// Two 8x8 b16 matrices; lanes 0-15 give the row addresses.
__device__ __forceinline__ void ldmatrix_x2(uint32_t (&r)[2], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n"
                 : "=r"(r[0]), "=r"(r[1])
                 : "r"(addr));
}

// 16-byte global->shared async copy; src_bytes in {0, 16} (0 = zero fill).
// Prefetch the line holding `p` into L2 (holds no registers while in flight).
__device__ __forceinline__ void prefetch_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];\n" ::"l"(p));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
                 "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// Streaming 16-byte global accesses for the read-modify-write of out.
// Eight consecutive 2-byte elements at p, which is only 2-byte aligned (rows
// of an odd-width matrix): the first nv of them (the rest read as zero), with
// the widest loads p's alignment allows (one 16-byte, two 8-byte, four
// 4-byte, or 2 + 4 + 4 + 4 + 2 bytes).  Never reads outside the nv elements.
// NC: the data is read-only for the kernel's lifetime (non-coherent path).
template <bool NC>
__device__ __forceinline__ uint4 ld8_u16(const uint16_t *p, int nv) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    if (nv >= 8) {
        if ((a & 15) == 0) return NC ? __ldg(reinterpret_cast<const uint4 *>(p)) : *reinterpret_cast<const uint4 *>(p);
        if ((a & 7) == 0) {
            const uint2 lo = NC ? __ldg(reinterpret_cast<const uint2 *>(p)) : *reinterpret_cast<const uint2 *>(p);
            const uint2 hi = NC ? __ldg(reinterpret_cast<const uint2 *>(p + 4)) : *reinterpret_cast<const uint2 *>(p + 4);
            return make_uint4(lo.x, lo.y, hi.x, hi.y);
        }
        const uint32_t *w = reinterpret_cast<const uint32_t *>(p + ((a & 3) ? 1 : 0));
        if ((a & 3) == 0) {
            return make_uint4(NC ? __ldg(w) : w[0], NC ? __ldg(w + 1) : w[1], NC ? __ldg(w + 2) : w[2],
                              NC ? __ldg(w + 3) : w[3]);
        }
        // elements 0 and 7 alone, pairs (1,2), (3,4), (5,6) as aligned words
        const uint32_t e0 = NC ? __ldg(p) : p[0], e7 = NC ? __ldg(p + 7) : p[7];
        const uint32_t w1 = NC ? __ldg(w) : w[0], w2 = NC ? __ldg(w + 1) : w[1], w3 = NC ? __ldg(w + 2) : w[2];
        return make_uint4(e0 | (w1 << 16), (w1 >> 16) | (w2 << 16), (w2 >> 16) | (w3 << 16),
                          (w3 >> 16) | (e7 << 16));
    }
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t lo = 2 * k < nv ? (NC ? __ldg(p + 2 * k) : p[2 * k]) : 0u;
        const uint32_t hi = 2 * k + 1 < nv ? (NC ? __ldg(p + 2 * k + 1) : p[2 * k + 1]) : 0u;
        w[k] = lo | (hi << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// The first nv of eight 2-byte elements (packed in v) to p, which is only
// 2-byte aligned, with the widest stores p's alignment allows.
__device__ __forceinline__ void st8_u16(uint16_t *p, uint4 v, int nv) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    if (nv >= 8) {
        if ((a & 15) == 0) {
            *reinterpret_cast<uint4 *>(p) = v;
        } else if ((a & 7) == 0) {
            reinterpret_cast<uint2 *>(p)[0] = make_uint2(v.x, v.y);
            reinterpret_cast<uint2 *>(p)[1] = make_uint2(v.z, v.w);
        } else if ((a & 3) == 0) {
            uint32_t *w = reinterpret_cast<uint32_t *>(p);
            w[0] = v.x;
            w[1] = v.y;
            w[2] = v.z;
            w[3] = v.w;
        } else {
            uint32_t *w = reinterpret_cast<uint32_t *>(p + 1);
            p[0] = (uint16_t)(v.x & 0xffffu);
            w[0] = (v.x >> 16) | (v.y << 16);
            w[1] = (v.y >> 16) | (v.z << 16);
            w[2] = (v.z >> 16) | (v.w << 16);
            p[7] = (uint16_t)(v.w >> 16);
        }
        return;
    }
    const uint32_t e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 8; ++k)
        if (k < nv) p[k] = (uint16_t)((e[k >> 1] >> (16 * (k & 1))) & 0xffffu);
}

__device__ __forceinline__ uint4 ld_global_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ void st_global_v4(void *p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};\n" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// ------------------------------------------------------------------ clusters
// Split cluster barrier (every thread of every CTA of the cluster arrives,
// then waits): release / acquire order each CTA's shared-memory accesses.
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
}
// Arrival without ordering this CTA's memory accesses (mbarrier
// initialisation is published by mbar_init's own fence).
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
// This CTA's rank within its cluster.
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
    return r;
}
// The shared::cluster address of `addr` (a shared::cta address) in CTA `rank`.
__device__ __forceinline__ uint32_t cluster_map(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
// Asynchronous 16-byte store into a cluster CTA's shared memory (`addr`)
// that counts its bytes on that CTA's mbarrier (`bar`), both shared::cluster
// addresses of the same CTA.
__device__ __forceinline__ void st_async_v4(uint32_t addr, float4 v, uint32_t bar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];\n" ::"r"(
            addr),
        "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(bar)
        : "memory");
}

// mbarrier in this CTA's shared memory, arrived at from the cluster.
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
// This CTA's arrival on its own mbarrier, announcing `bytes` of
// asynchronous stores for the current phase (they may land before or after).
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
// Bounded wait for phase `parity` of this CTA's mbarrier (acquire at cluster
// scope): false once kWaitPolls polls have failed.
constexpr int kWaitPolls = 1 << 20;
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t *bar, uint32_t parity) {
    const uint32_t addr = smem_u32(bar);
    for (int i = 0; i < kWaitPolls; ++i) {
        uint32_t ok;
        asm volatile(
            "{ .reg .pred p;\n"
            "  mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
            "  selp.u32 %0, 1, 0, p; }\n"
            : "=r"(ok)
            : "r"(addr), "r"(parity)
            : "memory");
        if (ok) return true;
    }
    return false;
}

// ------------------------------------------------------------------ tcgen05
// Fifth-generation tensor core: MMAs issued by one thread read both operands
// from shared memory (64-bit descriptors) and accumulate in tensor memory
// (TMEM), allocated per CTA in columns of 32-bit lanes x 128.

// Shared-memory descriptor of a K-major operand in the canonical 128-byte
// swizzled layout: rows of 128 bytes (64 fp16/bf16 of K), 8-row atoms of
// 1024 bytes (16-byte chunk c of row r at chunk c ^ (r & 7)), atoms stacked
// along M/N every 1024 bytes.  `addr`: shared address of the first row (an
// atom base, or an atom base + 32 * k for the k-th 16-wide K step).
__device__ __forceinline__ uint64_t tc_desc_sw128(uint32_t addr) {
    return (uint64_t)((addr & 0x3FFFF) >> 4)  // start address
           | (uint64_t)1 << 16                // leading byte offset (unused for this layout)
           | (uint64_t)(1024 >> 4) << 32      // stride byte offset: next 8-row atom
           | (uint64_t)1 << 46                // descriptor version
           | (uint64_t)2 << 61;               // 128-byte swizzle
}
// Instruction descriptor, kind::f16: fp32 accumulator, A and B both fp16 or
// both bf16, both K-major, M x N.
__host__ __device__ constexpr uint32_t tc_idesc_f16(bool bf16, int M, int N) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// One warp: allocate `ncols` (power of two >= 32) TMEM columns; the base
// address is written to shared memory at `slot`.
__device__ __forceinline__ void tc_alloc(uint32_t *slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                     smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tc_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
// D[taddr] (+)= A . B^T for one M x N x 16 step (accumulate: keep D).
__device__ __forceinline__ void tc_mma_f16(uint32_t taddr, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc, bool accumulate) {
    asm volatile(
        "{ .reg .pred p;\n"
        "  setp.ne.b32 p, %4, 0;\n"
        "  tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }\n" ::"r"(taddr),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate ? 1 : 0)
        : "memory");
}
// Arrive once on the mbarrier when this thread's earlier tcgen05 ops are done.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
                     smem_u32(bar))
                 : "memory");
}
// Warp-collective: this thread's TMEM lane (warp's lane quadrant + lane id),
// 16 consecutive 32-bit columns from `taddr`.
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15}, [%16];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// 32 consecutive 32-bit columns of this thread's TMEM lane, without waiting:
// the registers are valid only after tc_wait_ld().
__device__ __forceinline__ void tc_ld32_nowait(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tc_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}
// As tc_ld16 for 32 consecutive columns (one load, one wait).
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}
// Makes this thread's shared-memory writes (st.shared, cp.async) visible to
// the async proxy (tensor-core operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
// Bounded wait for phase `parity` of a CTA-local mbarrier: false once
// kWaitPolls polls have failed.
__device__ __forceinline__ bool mbar_wait_cta(uint64_t *bar, uint32_t parity) {
    const uint32_t addr = smem_u32(bar);
    for (int i = 0; i < kWaitPolls; ++i) {
        uint32_t ok;
        asm volatile(
            "{ .reg .pred p;\n"
            "  mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            "  selp.u32 %0, 1, 0, p; }\n"
            : "=r"(ok)
            : "r"(addr), "r"(parity)
            : "memory");
        if (ok) return true;
    }
    return false;
}

// ------------------------------------------------------------------ TMA
// Tiled 2-D tensor copy global -> this CTA's shared memory (cp.async.bulk.tensor):
// the box at (x = innermost element index, y = row) of the tensor map `map`
// (a __grid_constant__ kernel parameter) lands at `dst` in the map's swizzled
// layout; its bytes are counted on this CTA's mbarrier `bar`.  Elements
// outside the tensor are filled with zeros (and still counted).  x times the
// element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];\n" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}
// Tiled 3-D tensor copy global -> shared (as tma_load_2d, coordinates x, y, z).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            int z, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];\n" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}
// Tiled 2-D tensor copy this CTA's shared memory -> global: the box at (x, y)
// of `map` from `src` (laid out as a load of the same box would leave it);
// elements outside the tensor are not written.  Completion is tracked by the
// issuing thread's bulk async-groups (tma_store_commit / tma_store_wait_read).
// x times the element size must be a multiple of 16 bytes; x, y >= 0.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, int x, int y, uint32_t src) {
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];\n" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(x), "r"(y), "r"(src)
        : "memory");
}
__device__ __forceinline__ void tma_store_commit() {
    asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
}
// Waits until the issuing thread's committed bulk stores have finished
// reading their shared-memory source (they may still be writing to global).
__device__ __forceinline__ void tma_store_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory");
}
// Waits until the issuing thread's committed bulk stores are complete.
__device__ __forceinline__ void tma_store_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory");
}
// Starts fetching a tensor map (kernel parameter) into the descriptor cache.
__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Programmatic dependent launch: wait for the previous grid's results; let
// the next grid start launching.  Both are no-ops for an ordinary launch.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;\n"); }

// Plan entries outside their ranges (a token row outside [-1, T), an adapter
// id outside [-1, L), a tile row count outside [0, kTile]) are skipped by
// every build: the row reads as -1, the adapter as rank 0.  Builds with
// LORA_DEBUG defined also count them, as LORA_PLANERR_BOUNDS in the plan's
// error word (device-side bounds checks that neither trap nor stop).
__device__ __forceinline__ void plan_check_row(int row, int T, int32_t *hdr) {
#ifdef LORA_DEBUG
    if (row < -1 || row >= T) atomicOr(hdr + LORA_HDR_ERR, LORA_PLANERR_BOUNDS);
#else
    (void)row, (void)T, (void)hdr;
#endif
}
__device__ __forceinline__ void plan_check_tile(int4 tl, int L, int32_t *hdr) {
#ifdef LORA_DEBUG
    if (tl.x < -1 || tl.x >= L || tl.z < 0 || tl.z > kTile)
        atomicOr(hdr + LORA_HDR_ERR, LORA_PLANERR_BOUNDS);
#else
    (void)tl, (void)L, (void)hdr;
#endif
}

__device__ __forceinline__ int clamp_rank(const int32_t *ranks, int l, int R) {
    if (ranks == nullptr) return R;
    int r = __ldg(ranks + l);
    return r < 0 ? 0 : (r > R ? R : r);
}

// ------------------------------------------------------------------ block scan
// Exclusive prefix sum of one value per thread over the whole block
// (blockDim.x a multiple of 32, <= 1024).  `ws` holds >= 33 ints of shared
// memory.  Returns the exclusive prefix; *total receives the block sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int *ws, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    __syncthreads();
    if (lane == 31) ws[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nwarps ? ws[lane] : 0;
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int n = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += n;
        }
        if (lane < nwarps) ws[lane] = wi - w;
        if (lane == 31) ws[32] = wi;
    }
    __syncthreads();
    int res = ws[warp] + incl - v;
    *total = ws[32];
    return res;
}

// Exclusive prefix max of one value per thread over the block (same
// contract as block_exclusive_scan; the identity is INT_MIN).  *total
// receives the block maximum.
__device__ __forceinline__ int block_exclusive_max(int v, int *ws, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl = max(incl, n);
    }
    int excl = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) excl = INT_MIN;
    __syncthreads();
    if (lane == 31) ws[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nwarps ? ws[lane] : INT_MIN;
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int n = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi = max(wi, n);
        }
        int ex = __shfl_up_sync(0xffffffffu, wi, 1);
        if (lane == 0) ex = INT_MIN;
        if (lane < nwarps) ws[lane] = ex;
        if (lane == 31) ws[32] = wi;
    }
    __syncthreads();
    int res = max(ws[warp], excl);
    *total = ws[32];
    return res;
}

}  // namespace lora
