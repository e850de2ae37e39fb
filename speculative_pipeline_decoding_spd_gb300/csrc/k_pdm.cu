// Pipeline Draft Module kernels (run on the second stream, concurrently with the
// target's rounds).
//
// Speculative pipeline decoding, machine review "What carries the argument" / "Core
// claim": the module reads the pipeline's INPUT states, concatenates the target's
// hidden states at the anchor depths (deeper anchors of in-flight tokens are not yet
// computed and enter as zeros), projects them to one feature and runs Ls decoder layers
// and the LM head to propose the next token.  Its rows in one step are the token that
// left the pipeline last step (all anchors; its K,V stay in the module's cache) and
// the in-flight tokens, at consecutive positions, so its attention is plain causal
// attention over its own cache.
//
// Every GEMM here multiplies one weight matrix W [N][K] by R <= n+1 row vectors x [R][K]
// (a skinny GEMM: far more bytes of W than of x, so it is bound by streaming W once from
// HBM).  Design, one CTA per SM:
//   * a producer warp streams 8-row tiles of W (each row piece up to 6 KB, 1-D bulk copies)
//     into a shared-memory ring signalled by mbarriers, as the target's GEMVs do;
//   * the R rows of x are staged once per launch in shared memory as bf16 (or fp32 for
//     fp32 weights), with the input's normalisation / SiLU-product / anchor masking fused
//     into the staging;
//   * the 8 consumer warps split each tile's K range into 32-element blocks (block b to
//     warp b mod 8); per block a warp runs two m16n8k16 tensor-core steps with the x rows
//     as the 16-row A operand and the 8 weight rows as the B operand.  Both operands take
//     K in the same permuted order inside the block, so one 16-byte shared-memory read
//     per lane feeds a whole fragment;
//   * after the last K piece of a tile group the warps' partial 16x8 products meet in
//     shared memory and are added in warp order (deterministic), then the epilogue writes
//     or accumulates the outputs.
// A K range whose x rows do not fit in shared memory beside the ring is cut into slabs,
// one launch each; later slabs add into the output in slab order.
// RoPE and the append of the rows' K,V to the module's cache run in a small kernel
// between the QKV GEMM and attention (the rows' attention depends on one another's K,V).
#include "common.cuh"

namespace spd {

enum { OP_PROJ = 0, OP_QKV, OP_OPROJ, OP_GATEUP, OP_DOWN };

constexpr int PG_CONSUMERS = 256;              // 8 consumer warps
constexpr int PG_THREADS = PG_CONSUMERS + 32;  // + 1 producer warp
constexpr int PG_RG = 8;                       // weight rows per tile (the mma's n)
constexpr int PG_ROWB = 6144;                  // bytes of one row per tile piece, at most
constexpr int PG_MAXNS = 8;                    // ring stages at most
constexpr int PG_SMEM = 210 * 1024;            // x + reduction buffers + ring
constexpr int PG_XMAX = 96 * 1024;             // budget of the x rows of one slab
constexpr int PG_KB = 32;                      // K elements per warp block
constexpr int PG_BAR = 1;                      // named barrier of the consumer warps

__host__ __device__ inline int pg_round(int v, int m) { return (v + m - 1) / m * m; }
// row pitch (bytes) of x and of a weight tile: 128-byte multiple + 64, so the 8 rows that
// one fragment read touches fall alternately into the two halves of the banks
__host__ __device__ inline int pg_pitch(int elems, int esz) { return pg_round(elems * esz, 128) + 64; }
__host__ __device__ inline int pg_xbytes(int rows, int kx, int esz) { return pg_round(rows * pg_pitch(kx, esz), 128); }
__host__ __device__ inline int pg_redbytes(int MT) { return 2 * (PG_CONSUMERS / 32) * MT * 32 * 16; }
// K pieces of one slab of kw elements: nch pieces of KC elements (multiples of PG_KB)
__host__ __device__ inline int pg_nch(int kw, int esz) { return (kw * esz + PG_ROWB - 1) / PG_ROWB; }
__host__ __device__ inline int pg_kc(int kw, int esz) { return pg_round((kw + pg_nch(kw, esz) - 1) / pg_nch(kw, esz), PG_KB); }

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint4 lds128(const void *p) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(smem_u32(p)));
    return r;
}

template <int OP> __host__ __device__ inline int pg_N(const Plan &h) {
    return OP == OP_QKV ? h.qkv_rows : OP == OP_GATEUP ? 2 * h.F : h.d;
}
template <int OP> __host__ __device__ inline int pg_K(const Plan &h) {
    return OP == OP_PROJ ? h.nB * h.d : OP == OP_OPROJ ? h.q_rows : OP == OP_DOWN ? h.F : h.d;
}

// Weight rows of one GEMM: row u is row u of region 0 below b1, row u - b1 of region 1
// below b2, else row u - b2 of region 2.
template <typename T>
struct PgRows {
    const T *p0, *p1, *p2;
    int b1, b2, K;
    __device__ __forceinline__ const T *row(int u) const {
        if (u < b1) return p0 + (long long)u * K;
        if (u < b2) return p1 + (long long)(u - b1) * K;
        return p2 + (long long)(u - b2) * K;
    }
};
template <typename T, int OP>
__device__ __forceinline__ PgRows<T> pg_rows(const Plan *__restrict__ P, int layer, int K) {
    PgRows<T> r;
    r.K = K;
    r.b1 = r.b2 = 0x7fffffff;
    r.p1 = r.p2 = nullptr;
    if (OP == OP_PROJ) {
        r.p0 = reinterpret_cast<const T *>(P->proj);
        return r;
    }
    const LayerW &w = P->pl[layer];
    if (OP == OP_QKV) {
        r.p0 = reinterpret_cast<const T *>(w.wq);
        r.p1 = reinterpret_cast<const T *>(w.wk);
        r.p2 = reinterpret_cast<const T *>(w.wv);
        r.b1 = P->q_rows;
        r.b2 = P->q_rows + P->kv_rows;
    } else if (OP == OP_GATEUP) {
        r.p0 = reinterpret_cast<const T *>(w.wg);
        r.p1 = reinterpret_cast<const T *>(w.wu);
        r.b1 = P->F;
    } else {
        r.p0 = reinterpret_cast<const T *>(OP == OP_OPROJ ? w.wo : w.wd);
    }
    return r;
}

// ---- x staging (consumer warps only) ---------------------------------------------------
// x row r, slab-relative columns [0, kw): element k of the GEMM's input at k0 + k.
template <typename XT>
__device__ __forceinline__ void pg_store4(unsigned char *xs, int pitch, int r, int k, float4 v) {
    if (sizeof(XT) == 2) {
        __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t *>(&a);
        u.y = *reinterpret_cast<uint32_t *>(&b);
        *reinterpret_cast<uint2 *>(xs + r * pitch + k * 2) = u;
    } else {
        *reinterpret_cast<float4 *>(xs + r * pitch + k * 4) = v;
    }
}

// Per-row RMS statistics of Xp rows 0..R-1 from the per-CTA sums of squares that the
// kernel which last wrote Xp left in ssp (CTA order, then a fixed shuffle tree).
__device__ __noinline__ void pg_row_inv_rms(const Plan *__restrict__ P, int R, float *inv) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, G = P->pdm_grid;
    for (int r = warp; r < R; r += PG_CONSUMERS / 32) {
        float s = 0.f;
        for (int c = lane; c < G; c += 32) s += P->ssp[c * MAXS + r];
        s = warp_sum(s);
        if (lane == 0) inv[r] = 1.0f / sqrtf(s / (float)P->d + P->eps);
    }
}

// Stage the slab of all R rows: items are 4-element groups, 8 in flight per thread.
template <typename XT, int OP>
__device__ __noinline__ void pg_stage_x(const Plan *__restrict__ P, const PdmRows &pr, int layer, int k0, int kw,
                                        unsigned char *xs, int pitch, const float *inv) {
    const int R = pr.R, kw4 = kw >> 2, total = R * kw4, d = P->d;
    const float *g = OP == OP_QKV ? P->pl[layer].g1 : OP == OP_GATEUP ? P->pl[layer].g2 : nullptr;
    for (int b = threadIdx.x; b < total; b += 8 * PG_CONSUMERS) {
        float4 v[8], w[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = b + u * PG_CONSUMERS;
            if (i >= total) continue;
            const int r = i / kw4, k = k0 + 4 * (i - r * kw4);
            if (OP == OP_PROJ) {
                const int a = k / d, off = k - a * d;
                v[u] = P->anchors[a] <= pr.depth[r]
                           ? *reinterpret_cast<const float4 *>(P->ANCH + ((long long)pr.slot[r] * P->nB + a) * d + off)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
            } else if (OP == OP_QKV || OP == OP_GATEUP) {
                v[u] = *reinterpret_cast<const float4 *>(P->Xp + (long long)r * d + k);
                w[u] = *reinterpret_cast<const float4 *>(g + k);
            } else if (OP == OP_OPROJ) {
                v[u] = *reinterpret_cast<const float4 *>(P->ATTp + (long long)r * P->q_rows + k);
            } else {
                v[u] = *reinterpret_cast<const float4 *>(P->GUp + (long long)r * 2 * P->F + k);
                w[u] = *reinterpret_cast<const float4 *>(P->GUp + (long long)r * 2 * P->F + P->F + k);
            }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = b + u * PG_CONSUMERS;
            if (i >= total) continue;
            const int r = i / kw4, kk = 4 * (i - r * kw4);
            float4 x = v[u];
            if (OP == OP_QKV || OP == OP_GATEUP) {
                const float s = inv[r];
                x = make_float4((x.x * s) * w[u].x, (x.y * s) * w[u].y, (x.z * s) * w[u].z, (x.w * s) * w[u].w);
            } else if (OP == OP_DOWN) {
                x = make_float4(silu_f(x.x) * w[u].x, silu_f(x.y) * w[u].y, silu_f(x.z) * w[u].z, silu_f(x.w) * w[u].w);
            }
            pg_store4<XT>(xs, pitch, r, kk, x);
        }
    }
}

// ---- the GEMM ---------------------------------------------------------------------------
// Output rows [lo, hi) of this CTA in groups of 8; slab [k0, k0 + kw) of K, kw = min(kx, K - k0).
template <typename T, int OP, int MT>
__global__ void __launch_bounds__(PG_THREADS, 1) k_pdm_gemm(const Plan *__restrict__ P, int layer, int k0, int kx) {
    using XT = T;   // x rows are kept in the weights' type (bf16 operands for the tensor cores)
    constexpr int ESZ = sizeof(T);
    extern __shared__ __align__(128) unsigned char pg_smem[];
    __shared__ __align__(8) uint64_t full[PG_MAXNS], empty[PG_MAXNS];
    __shared__ PdmRows pr;
    __shared__ float s_inv[MAXS];
    __shared__ int s_done;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (warp == 0) {
        warp_pdm_rows(P, pr, &s_done);
        if (lane == 0) {
            for (int i = 0; i < PG_MAXNS; ++i) {
                mbar_init(&full[i], 1);
                mbar_init(&empty[i], PG_CONSUMERS / 32);
            }
            fence_mbar_init();
        }
    }
    __syncthreads();
    if (s_done || pr.R < 1) return;

    const int N = pg_N<OP>(*P), K = pg_K<OP>(*P);
    const int kw = min(kx, K - k0);
    const int nch = pg_nch(kw, ESZ), KC = pg_kc(kw, ESZ);
    const int xpitch = pg_pitch(kx, ESZ);
    const int rowb = pg_pitch(KC, ESZ), stage_bytes = PG_RG * rowb;
    const int xbytes = pg_xbytes(P->n + 1, kx, ESZ);
    unsigned char *xs = pg_smem;
    float4 *red = reinterpret_cast<float4 *>(pg_smem + xbytes);
    unsigned char *stages = pg_smem + xbytes + pg_redbytes(MT);
    const int NS = min(PG_MAXNS, (PG_SMEM - xbytes - pg_redbytes(MT)) / stage_bytes);
    const int lo = (int)((long long)N * blockIdx.x / gridDim.x);
    const int hi = (int)((long long)N * (blockIdx.x + 1) / gridDim.x);

    if (warp == PG_CONSUMERS / 32) {
        // ------------------------------ producer ----------------------------------------
        if (lane == 0) {
            const PgRows<T> wr = pg_rows<T, OP>(P, layer, K);
            uint32_t tile = 0;
            for (int g0 = lo; g0 < hi; g0 += PG_RG) {
                const T *rp[PG_RG];
                int nrows = 0;
#pragma unroll
                for (int q = 0; q < PG_RG; ++q) {
                    rp[q] = g0 + q < hi ? wr.row(g0 + q) + k0 : nullptr;
                    nrows += rp[q] != nullptr;
                }
                for (int c = 0; c < nch; ++c) {
                    const int kc0 = c * KC, len = min(KC, kw - kc0);
                    const int sidx = tile % NS;
                    const uint32_t u = tile / NS;
                    if (!mbar_wait(&empty[sidx], (u & 1) ^ 1)) P->st->error = ERR_TIMEOUT;
                    const uint32_t bytes = (uint32_t)len * ESZ;
                    mbar_expect_tx(&full[sidx], bytes * nrows);
#pragma unroll
                    for (int q = 0; q < PG_RG; ++q)
                        if (rp[q]) bulk_g2s(stages + sidx * stage_bytes + q * rowb, rp[q] + kc0, bytes, &full[sidx]);
                    ++tile;
                }
            }
        }
        return;
    }

    // ------------------------------ consumers -------------------------------------------
    const int tid = threadIdx.x, R = pr.R;
    if (OP == OP_QKV || OP == OP_GATEUP) {
        pg_row_inv_rms(P, R, s_inv);
        named_sync(PG_BAR, PG_CONSUMERS);
    }
    pg_stage_x<XT, OP>(P, pr, layer, k0, kw, xs, xpitch, s_inv);
    named_sync(PG_BAR, PG_CONSUMERS);

    // output of one (x row, weight row) pair
    const int d = P->d;
    float *dst;
    int ld;
    bool accum;
    if (OP == OP_QKV) {
        dst = P->QKVp; ld = P->qkv_rows; accum = k0 > 0;
    } else if (OP == OP_GATEUP) {
        dst = P->GUp; ld = 2 * P->F; accum = k0 > 0;
    } else {
        dst = P->Xp; ld = d; accum = OP != OP_PROJ || k0 > 0;
    }

    // kernels that finish an Xp row (the last slab of proj / o / down) leave per-CTA sums of
    // squares for the next normalisation; reduction thread t always owns the same
    // (x row, weight row) pair of a group, so it sums its squares over the groups in order
    const bool want_ss = (OP == OP_PROJ || OP == OP_OPROJ || OP == OP_DOWN) && k0 + kw == K;
    float sq = 0.f;
    const int gq = lane >> 2, tq = lane & 3;
    uint32_t tile = 0;
    int buf = 0;
    for (int g0 = lo; g0 < hi; g0 += PG_RG) {
        // bf16: acc[4m..4m+3] is the m-th 16x8 mma accumulator fragment; fp32: acc[j] is the
        // (x row (lane >> 3) + 4j, weight row lane & 7) product
        float acc[4 * MT];
#pragma unroll
        for (int j = 0; j < 4 * MT; ++j) acc[j] = 0.f;
        for (int c = 0; c < nch; ++c) {
            const int kc0 = c * KC, len = min(KC, kw - kc0), nblk = len / PG_KB;
            const int sidx = tile % NS;
            const uint32_t u = tile / NS;
            if (!mbar_wait(&full[sidx], u & 1)) P->st->error = ERR_TIMEOUT;
            const unsigned char *tb = stages + sidx * stage_bytes;
            if constexpr (ESZ == 2) {
                // lane (gq, tq): weight row gq, x rows gq and gq + 8 (+16 m), elements 8tq..8tq+7 of
                // each 32-block; the two mma steps take elements {8tq..8tq+3} and {8tq+4..8tq+7}
                const unsigned char *wp = tb + gq * rowb + tq * 16;
                const unsigned char *xp = xs + gq * xpitch + kc0 * 2 + tq * 16;
                bool xv[MT][2];
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    xv[m][0] = m * 16 + gq < R;
                    xv[m][1] = m * 16 + 8 + gq < R;
                }
                // the two mma steps of a block go to two accumulator chains (added at the end of
                // the piece, fixed order)
                float acc2[4 * MT];
#pragma unroll
                for (int j = 0; j < 4 * MT; ++j) acc2[j] = 0.f;
                for (int b = warp; b < nblk; b += PG_CONSUMERS / 32) {
                    const uint4 w = lds128(wp + b * 64);
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                        const uint4 xa = xv[m][0] ? lds128(xp + (m * 16) * xpitch + b * 64) : z;
                        const uint4 xb = xv[m][1] ? lds128(xp + (m * 16 + 8) * xpitch + b * 64) : z;
                        float(&f)[4] = *reinterpret_cast<float(*)[4]>(&acc[4 * m]);
                        float(&f2)[4] = *reinterpret_cast<float(*)[4]>(&acc2[4 * m]);
                        mma_bf16(f, xa.x, xb.x, xa.y, xb.y, w.x, w.y);
                        mma_bf16(f2, xa.z, xb.z, xa.w, xb.w, w.z, w.w);
                    }
                }
#pragma unroll
                for (int j = 0; j < 4 * MT; ++j) acc[j] += acc2[j];
            } else {
                // fp32 weights: plain FMAs in element order
                const int wrow = lane & 7, xq = lane >> 3;
                const float *wp = reinterpret_cast<const float *>(tb + wrow * rowb);
                for (int b = warp; b < nblk; b += PG_CONSUMERS / 32) {
                    for (int e = 0; e < PG_KB; ++e) {
                        const int k = b * PG_KB + e;
                        const float wv = wp[k];
#pragma unroll
                        for (int j = 0; j < 4 * MT; ++j) {
                            const int xr = xq + 4 * j;
                            if (xr < R) acc[j] = fmaf(wv, reinterpret_cast<const float *>(xs + xr * xpitch)[kc0 + k], acc[j]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[sidx]);
            ++tile;
        }
        // ---- partial products of all warps -> fixed-order sum -> epilogue
        // shared buffer in the mma fragment layout: [buf][warp][m][lane] x 4 floats, float
        // (m, lane, reg) = product (x row 16m + 8(reg >> 1) + lane / 4, weight row 2(lane % 4) + reg % 2)
        if constexpr (ESZ == 2) {
#pragma unroll
            for (int m = 0; m < MT; ++m)
                red[((buf * (PG_CONSUMERS / 32) + warp) * MT + m) * 32 + lane] =
                    make_float4(acc[4 * m], acc[4 * m + 1], acc[4 * m + 2], acc[4 * m + 3]);
        } else {
            float *rf = reinterpret_cast<float *>(red);
            const int wrow = lane & 7, xq = lane >> 3;
#pragma unroll
            for (int j = 0; j < 4 * MT; ++j) {
                const int xr = xq + 4 * j, m = xr >> 4, r16 = xr & 15;
                const int l2 = (r16 & 7) * 4 + (wrow >> 1), reg = (r16 >> 3) * 2 + (wrow & 1);
                rf[(((buf * (PG_CONSUMERS / 32) + warp) * MT + m) * 32 + l2) * 4 + reg] = acc[j];
            }
        }
        named_sync(PG_BAR, PG_CONSUMERS);
        if (tid < 128 * MT) {
            const int m = tid >> 7, l = (tid >> 2) & 31, reg = tid & 3;
            const float *rf = reinterpret_cast<const float *>(red);
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < PG_CONSUMERS / 32; ++w) s += rf[(((buf * (PG_CONSUMERS / 32) + w) * MT + m) * 32 + l) * 4 + reg];
            const int xr = m * 16 + (reg >> 1) * 8 + (l >> 2);
            const int row = g0 + (l & 3) * 2 + (reg & 1);
            if (xr < R && row < hi) {
                float *o = dst + (long long)xr * ld + row;
                const float v = accum ? *o + s : s;
                *o = v;
                sq = fmaf(v, v, sq);
            }
        }
        buf ^= 1;
    }
    if (want_ss && tid < 128 * MT) {
        // the 8 weight rows of one x row sit in lanes differing in bits 0, 2 and 3 of tid
        sq += __shfl_xor_sync(0xffffffffu, sq, 1);
        sq += __shfl_xor_sync(0xffffffffu, sq, 4);
        sq += __shfl_xor_sync(0xffffffffu, sq, 8);
        const int m = tid >> 7, l = (tid >> 2) & 31, reg = tid & 3;
        if ((tid & 13) == 0) P->ssp[blockIdx.x * MAXS + m * 16 + (reg >> 1) * 8 + (l >> 2)] = sq;
    }
}

// ---- RoPE of q and k, and the rows' K,V into the module's cache ---------------------------
template <typename T>
__global__ void __launch_bounds__(256) k_pdm_rope_kv(const Plan *__restrict__ P, int layer) {
    __shared__ PdmRows pr;
    __shared__ int s_done;
    if (threadIdx.x < 32) warp_pdm_rows(P, pr, &s_done);
    __syncthreads();
    const int r = blockIdx.x;
    if (s_done || r >= pr.R) return;
    // items: q pairs, k pairs (rotate-half RoPE at the row's position), then v elements
    const int hd = P->hd, half = hd >> 1, pos = pr.pos0 + r;
    const int nq = P->Hq * half, nk = P->Hkv * half, i = blockIdx.y * blockDim.x + threadIdx.x;
    if (i >= nq + nk + P->kv_rows) return;
    float *q = P->QKVp + (long long)r * P->qkv_rows;
    const long long off = (long long)layer * P->kv_stride + (long long)pos * P->kv_rows;
    if (i < nq + nk) {
        const int ii = i < nq ? i : i - nq;
        const int h = ii / half, j = ii - h * half;
        float *src = (i < nq ? q : q + P->q_rows) + h * hd + j;
        const float2 c = P->rope[(long long)pos * half + j];
        const float a = src[0], b = src[half];
        const float y0 = a * c.x - b * c.y, y1 = b * c.x + a * c.y;
        if (i < nq) {
            src[0] = y0;
            src[half] = y1;
        } else {
            T *kc = reinterpret_cast<T *>(P->pkc) + off + h * hd + j;
            kc[0] = WTraits<T>::store(y0);
            kc[half] = WTraits<T>::store(y1);
        }
    } else {
        const int e = i - nq - nk;
        reinterpret_cast<T *>(P->pvc)[off + e] = WTraits<T>::store(q[P->q_rows + P->kv_rows + e]);
    }
}

// ---------------------------------------------------------------------------------
// Host side: slab width per GEMM so that the x rows of one slab fit their budget.
static int pg_slab(int K, int rows, int esz) {
    int kx = pg_round(K, PG_KB);
    int ns = 1;
    while (pg_xbytes(rows, kx, esz) > PG_XMAX) {
        ++ns;
        kx = pg_round((K + ns - 1) / ns, PG_KB);
    }
    return kx;
}

void pdm_plan(const Plan &h, PdmPlan &pp) {
    const int esz = h.dtype == SPD_BF16 ? 2 : 4, rows = h.n + 1;
    pp.MT = rows <= 16 ? 1 : 2;
    const int Ks[5] = {pg_K<OP_PROJ>(h), pg_K<OP_QKV>(h), pg_K<OP_OPROJ>(h), pg_K<OP_GATEUP>(h), pg_K<OP_DOWN>(h)};
    for (int i = 0; i < 5; ++i) {
        pp.kx[i] = pg_slab(Ks[i], rows, esz);
        pp.ns[i] = (Ks[i] + pp.kx[i] - 1) / pp.kx[i];
    }
}

template <typename T, int OP, int MT>
static void pg_launch(const Plan *P, const Plan &h, const PdmPlan &pp, int layer, int grid, cudaStream_t s) {
    const int K = pg_K<OP>(h), kx = pp.kx[OP];
    for (int k0 = 0; k0 < K; k0 += kx) k_pdm_gemm<T, OP, MT><<<grid, PG_THREADS, PG_SMEM, s>>>(P, layer, k0, kx);
}

template <typename T, int MT>
static void pdm_step_mt(const Plan *P, const Plan &h, const PdmPlan &pp, int grid, cudaStream_t s) {
    pg_launch<T, OP_PROJ, MT>(P, h, pp, 0, grid, s);
    for (int li = 0; li < h.Ls; ++li) {
        pg_launch<T, OP_QKV, MT>(P, h, pp, li, grid, s);
        const int items = (h.Hq + h.Hkv) * (h.hd / 2) + h.kv_rows;
        k_pdm_rope_kv<T><<<dim3(h.n + 1, (items + 255) / 256), 256, 0, s>>>(P, li);
        launch_pdm_attn<T>(P, h, li, s);
        pg_launch<T, OP_OPROJ, MT>(P, h, pp, li, grid, s);
        pg_launch<T, OP_GATEUP, MT>(P, h, pp, li, grid, s);
        pg_launch<T, OP_DOWN, MT>(P, h, pp, li, grid, s);
    }
}

template <typename T>
void launch_pdm_step(const Plan *P, const Plan &h, const PdmPlan &pp, int grid, cudaStream_t s) {
    if (pp.MT == 1) pdm_step_mt<T, 1>(P, h, pp, grid, s);
    else pdm_step_mt<T, 2>(P, h, pp, grid, s);
}

template <typename T, int MT>
static void set_attr_mt() {
    cudaFuncSetAttribute(k_pdm_gemm<T, OP_PROJ, MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, PG_SMEM);
    cudaFuncSetAttribute(k_pdm_gemm<T, OP_QKV, MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, PG_SMEM);
    cudaFuncSetAttribute(k_pdm_gemm<T, OP_OPROJ, MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, PG_SMEM);
    cudaFuncSetAttribute(k_pdm_gemm<T, OP_GATEUP, MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, PG_SMEM);
    cudaFuncSetAttribute(k_pdm_gemm<T, OP_DOWN, MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, PG_SMEM);
}

void set_pdm_attributes() {
    set_attr_mt<float, 1>();
    set_attr_mt<float, 2>();
    set_attr_mt<__nv_bfloat16, 1>();
    set_attr_mt<__nv_bfloat16, 2>();
}

template void launch_pdm_step<float>(const Plan *, const Plan &, const PdmPlan &, int, cudaStream_t);
template void launch_pdm_step<__nv_bfloat16>(const Plan *, const Plan &, const PdmPlan &, int, cudaStream_t);

}  // namespace spd
