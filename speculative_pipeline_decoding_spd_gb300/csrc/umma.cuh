// Dense bf16 GEMM on the fifth-generation tensor cores (tcgen05 / TMEM / TMA), used by the
// prefill, the one place on the path where a tile really is a dense contraction: a chunk
// of prompt rows times every weight matrix of every layer (machine review, "What carries
// the argument": the prefill must leave every layer's K,V and the draft module's
// full-depth prefix).
//
//   C[M][N]  =  or  +=  (A_hi + A_lo)[M][K] . W[N][K]^T
//
// A is an fp32 activation given as two bf16 parts (hi = bf16(a), lo = bf16(a - hi)), so
// the products see about 16 mantissa bits of the activation; W is a bf16 weight matrix
// in its [out][in] layout (K-major, as the tensor cores take both operands).  One CTA
// computes one 128 x BN tile of C with fp32 accumulation in tensor memory:
//   * warp 4, one lane: TMA loads of the K blocks (64 wide) of A_hi, A_lo and W into a
//     ring of shared-memory stages (128-byte swizzle), signalled by mbarriers;
//   * warp 5, one lane: tcgen05.mma (M 128, N BN, K 16), two per K step (A_hi and A_lo
//     against the same W tile); tcgen05.commit frees a stage when its MMAs are done and,
//     after the last block, signals the accumulator; warp 5 also allocates and frees the
//     BN tensor-memory columns;
//   * warps 0-3: the epilogue, each reading its 32 lanes (rows) of the accumulator with
//     tcgen05.ld and storing (or adding into) fp32 C.
// Every wait is bounded; a wait that runs out sets *err (the run state's error word) and
// the kernel carries on to its end, where the tensor memory is freed.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace spd {

constexpr int UM_BM = 128;                 // rows of a tile (the MMA's M)
constexpr int UM_BK = 64;                  // K per stage: one 128-byte swizzle row of bf16
constexpr int UM_THREADS = 192;            // 4 epilogue warps, TMA warp, MMA warp
constexpr int UM_SMEM = 200 * 1024 + 1024; // stages + alignment slack
constexpr int UM_A_BYTES = UM_BM * UM_BK * 2;

template <int BN> __host__ __device__ constexpr int um_stage_bytes() { return 2 * UM_A_BYTES + BN * UM_BK * 2; }
template <int BN> __host__ __device__ constexpr int um_stages() {
    return (UM_SMEM - 1024) / um_stage_bytes<BN>() > 6 ? 6 : (UM_SMEM - 1024) / um_stage_bytes<BN>();
}

struct UmmaArgs {
    float *C;
    int ldc;          // row pitch of C (floats)
    int M, N, K;      // rows of A and C, columns of C, reduction length (multiple of 64)
    int a_lo_row;     // first row of the A_lo part in A's tensor map (A_hi starts at row 0)
    int accumulate;   // 1: C += result (the residual stream), 0: C = result
    int *err;         // error word of the run state (ERR_TIMEOUT on a wait that ran out)
};

// ---- PTX wrappers -------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// whole warp: allocate ncols (a power of two >= 32) tensor-memory columns; the base address
// is written to *dst in shared memory
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_free(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// D[tmem] (+)= A[smem desc] . B[smem desc]^T, bf16 inputs, fp32 accumulator
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// arrive once on bar when every tcgen05 operation this thread issued so far has completed
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
// 16 consecutive fp32 columns of this thread's lane
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major tile written by TMA with 128-byte swizzle:
// rows of 128 bytes (64 bf16 of K), 8-row swizzle atoms 1024 bytes apart (stride byte
// offset), leading byte offset unused for this layout (1), descriptor version 1, layout
// type 2 (128-byte swizzle).  Moving to the next 16-element K step inside the 128-byte
// row adds 32 bytes to the start address.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3ffffu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor, kind::f16: fp32 accumulator (bits 4-5 = 1), A and B bf16 (bits
// 7-9 and 10-12 = 1), both K-major (bits 15, 16 = 0), N / 8 at bits 17-22, M / 16 at 24-28.
__host__ __device__ constexpr uint32_t umma_idesc(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

template <int BN>
__global__ void __launch_bounds__(UM_THREADS, 1)
    k_umma_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW, UmmaArgs a) {
    constexpr int SB = um_stage_bytes<BN>(), NS = um_stages<BN>();
    extern __shared__ uint8_t um_smem[];
    __shared__ __align__(8) uint64_t full[NS], empty[NS], accb;
    __shared__ uint32_t s_tmem;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * BN, m0 = blockIdx.y * UM_BM, nk = a.K / UM_BK;
    const uint32_t base = (smem_u32(um_smem) + 1023u) & ~1023u;   // 1024-byte aligned stages
    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(&accb, 1);
        fence_mbar_init();
    }
    if (warp == 4 && lane == 0) {
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmW);
    }
    if (warp == 5) tmem_alloc(&s_tmem, BN);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    bool timed_out = false;

    if (warp == 4) {
        if (lane == 0) {
            // ---- TMA producer
            for (int kb = 0; kb < nk; ++kb) {
                const int s = kb % NS;
                const uint32_t u = (uint32_t)(kb / NS);
                if (!mbar_wait(&empty[s], (u & 1) ^ 1)) timed_out = true;
                mbar_expect_tx(&full[s], SB);
                const uint32_t sa = base + s * SB;
                tma_load_2d(sa, &tmA, kb * UM_BK, m0, &full[s]);
                tma_load_2d(sa + UM_A_BYTES, &tmA, kb * UM_BK, a.a_lo_row + m0, &full[s]);
                tma_load_2d(sa + 2 * UM_A_BYTES, &tmW, kb * UM_BK, n0, &full[s]);
            }
            // the last copies into each stage have landed before the CTA can exit (the MMA
            // issuer waits for them too, unless one of its waits ran out)
            for (int kb = nk > NS ? nk - NS : 0; kb < nk; ++kb)
                if (!mbar_wait(&full[kb % NS], (uint32_t)(kb / NS) & 1)) timed_out = true;
        }
    } else if (warp == 5) {
        if (lane == 0) {
            // ---- MMA issuer
            constexpr uint32_t idesc = umma_idesc(UM_BM, BN);
            for (int kb = 0; kb < nk; ++kb) {
                const int s = kb % NS;
                const uint32_t u = (uint32_t)(kb / NS);
                if (!mbar_wait(&full[s], u & 1)) timed_out = true;
                tc_fence_after();
                const uint32_t sa = base + s * SB;
#pragma unroll
                for (int k = 0; k < UM_BK / 16; ++k) {
                    const uint64_t bd = umma_desc(sa + 2 * UM_A_BYTES + 32 * k);
                    umma_bf16(tmem, umma_desc(sa + 32 * k), bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
                    umma_bf16(tmem, umma_desc(sa + UM_A_BYTES + 32 * k), bd, idesc, 1u);
                }
                umma_commit(&empty[s]);
            }
            umma_commit(&accb);
        }
    } else {
        // ---- epilogue: warp w reads accumulator lanes 32w..32w+31 (its rows)
        if (!mbar_wait(&accb, 0)) timed_out = true;
        tc_fence_after();
        const int row = m0 + warp * 32 + lane;
        float *crow = a.C + (long long)row * a.ldc + n0;
        for (int c = 0; c < BN; c += 16) {
            uint32_t r[16];
            tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c, r);
            if (row < a.M) {
                float4 *cp = reinterpret_cast<float4 *>(crow + c);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float4 v = make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                           __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
                    if (a.accumulate) {
                        const float4 o = cp[q];
                        v.x += o.x;
                        v.y += o.y;
                        v.z += o.z;
                        v.w += o.w;
                    }
                    cp[q] = v;
                }
            }
        }
    }
    if (timed_out) *a.err = ERR_TIMEOUT;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 5) tmem_free(tmem, BN);
}

}  // namespace spd
