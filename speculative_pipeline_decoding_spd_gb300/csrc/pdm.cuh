// Draft-module GEMM, CTA-level device code of the draft kernels (k_pdm.cu).
//
// Speculative pipeline decoding, machine review "What carries the argument" / "Core
// claim": the draft module reads the pipeline's INPUT states, concatenates the target's
// hidden states at the anchor depths (deeper anchors of in-flight tokens are not yet
// computed and enter as zeros), projects them to one feature and runs Ls decoder layers.
// Its rows in one step are the token that left the pipeline last step and the in-flight
// tokens, at consecutive positions.
//
// Every GEMM here multiplies one weight matrix W [N][K] by R <= n+1 row vectors x [R][K]
// (far more bytes of W than of x: bound by streaming W once from HBM).  With bf16 weights
// each x row arrives as two bf16 rows, hi = bf16(x) and lo = bf16(x - hi), and both meet the
// weights on the tensor cores (the products add up in the same accumulators), so the GEMM
// sees x at about 16 mantissa bits, not 8.  (In fp64 on the 4B shape over 8 decode steps,
// rounding one kind of input to bf16 moves the newest row's draft logits by 1.7e-2 (gate/up),
// 1.6e-2 (O), 1.3e-2 (down), 3.8e-3 (QKV), 0.7e-3 (projection); all of them 2.7e-2.)  A group
// of CTAs does one GEMM; per CTA:
//   * a producer warp streams 8-row tiles of W (each row piece up to 6 KB, 1-D bulk
//     copies) into a shared-memory ring signalled by mbarriers;
//   * the R rows of x for the CTA's K slab go to shared memory: for bf16 weights the kernel
//     before left them as bf16 rows in global memory and one thread copies them with bulk
//     copies (the projection per anchor, deeper anchors zeroed); for fp32 weights the
//     consumer warps load and stage them with the norm weight / anchor masking fused in.
//     An RMS-normalised input is x * g, and its row's 1/rms (a per-row scalar) scales the
//     GEMM's output instead, so staging does not wait for the row statistics;
//   * the 8 consumer warps split each tile's K range into 32-element blocks (block b to
//     warp b mod 8); per block a warp runs two m16n8k16 tensor-core steps with the x rows
//     as the 16-row A operand and the 8 weight rows as the B operand, both taking K in the
//     same permuted order inside the block, so one 16-byte shared-memory read per lane
//     feeds a whole fragment;
//   * after the last K piece of a tile group the warps' partial 16x8 products meet in
//     shared memory and are added in warp order, then the epilogue finishes the outputs.
// The CTAs of a GEMM split its output rows into row blocks and, when the x rows of all of
// K do not fit in shared memory, its K range into ns slabs: CTA p works on row block
// p / ns, slab p % ns.  Slab CTAs leave partial sums; the last to arrive at a row block
// adds them in slab order and finishes the outputs.
// Epilogues: the QKV GEMM applies RoPE and appends the rows' K,V to the module's cache
// (a tile holds 4 rotary pairs: rows i and i + hd/2 of one head, so both halves meet in
// one warp); gate/up tiles likewise hold gate rows u..u+3 with up rows F+u..F+u+3, and the
// epilogue leaves SiLU(gate) * up, the down GEMM's input; projection, O and down finish
// residual rows and leave per-8-row sums of squares for the next normalisation
// (independent of how CTAs split the work).
#pragma once

#include "common.cuh"

namespace spd {

enum { OP_PROJ = 0, OP_QKV, OP_OPROJ, OP_GATEUP, OP_DOWN, OP_LM };

constexpr int PG_CONSUMERS = 256;              // 8 consumer warps
constexpr int PG_THREADS = PG_CONSUMERS + 32;  // + 1 producer warp
constexpr int PG_RG = 8;                       // weight rows per tile (the mma's n)
constexpr int PG_ROWB = 6144;                  // bytes of one row per tile piece, at most
constexpr int PG_MAXNS = 8;                    // ring stages at most
constexpr int PG_SMEM = 224 * 1024;            // x + reduction buffers + ring
constexpr int PG_XMAX = 96 * 1024;             // budget of the x rows (both parts) of one slab
constexpr int PG_XRB = 10;                     // register-resident x: 32-element blocks per warp, at most
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

template <int OP> __host__ __device__ inline int pg_N(const Plan &h) {
    return OP == OP_QKV ? h.qkv_rows : OP == OP_GATEUP ? 2 * h.F : OP == OP_LM ? h.V : h.d;
}
template <int OP> __host__ __device__ inline int pg_K(const Plan &h) {
    return OP == OP_PROJ ? h.nB * h.d : OP == OP_OPROJ ? h.q_rows : OP == OP_DOWN ? h.F : h.d;
}

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
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(smem_u32(p)));
    return r;
}

// Weight rows of one draft GEMM.  Output row of tile slot q in group g: 8g + q, except for
// the q and k rows of the QKV GEMM, where group g holds rotary pairs 4g .. 4g+3 (pair u =
// (head u / (hd/2), element u mod (hd/2))): slots 0..3 the first halves, 4..7 the second.
template <typename T, int OP>
struct PgRows {
    const T *p0, *p1, *p2;
    int b1, b2, K, hd, qk_groups;
    __device__ __forceinline__ int row_of(int g, int q) const {
        if (OP == OP_QKV && g < qk_groups) {
            const int half = hd >> 1, u = 4 * g + (q & 3), h = u / half;
            return h * hd + (u - h * half) + (q >= 4 ? half : 0);
        }
        if (OP == OP_GATEUP) return 4 * g + (q & 3) + (q >= 4 ? b1 : 0);   // gate rows u, up rows F + u
        return 8 * g + q;
    }
    __device__ __forceinline__ const T *ptr(int row) const {
        if (row < b1) return p0 + (long long)row * K;
        if (row < b2) return p1 + (long long)(row - b1) * K;
        return p2 + (long long)(row - b2) * K;
    }
};
template <typename T, int OP>
__device__ __forceinline__ PgRows<T, OP> pg_rows(const Plan *__restrict__ P, int layer) {
    PgRows<T, OP> r;
    r.K = pg_K<OP>(*P);
    r.hd = P->hd;
    r.qk_groups = (P->q_rows + P->kv_rows) / 8;
    r.b1 = r.b2 = 0x7fffffff;
    r.p1 = r.p2 = nullptr;
    if (OP == OP_PROJ || OP == OP_LM) {
        r.p0 = reinterpret_cast<const T *>(OP == OP_PROJ ? P->proj : P->lm_head);
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

// Draft GEMMs whose bf16 input rows come as hi and lo parts: all but the LM head (whose four
// rows carry both parts of its two rows already).
template <int OP> __host__ __device__ constexpr bool pg_hilo() { return OP != OP_LM; }

// bf16 input row element in two parts: hi at p[i], lo (what hi left out) at p[lo_off + i]
__device__ __forceinline__ void store_hilo(__nv_bfloat16 *p, long long lo_off, long long i, float v) {
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    p[i] = hi;
    p[lo_off + i] = __float2bfloat16_rn(v - __bfloat162float(hi));
}

// ---- x staging (consumer warps only) ---------------------------------------------------
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

// Per-row RMS statistics of Xp rows 0..R-1 from the per-8-row sums of squares that the GEMM
// which last finished Xp left in ssp [row][d / 8] (lane-strided in order, then a fixed
// shuffle tree); each lane's loads of a row are issued together.
static __device__ __noinline__ void pg_row_inv_rms(const Plan *__restrict__ P, int R, float *inv) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, ng = P->d / 8;
    for (int r = warp; r < R; r += PG_CONSUMERS / 32) {
        const float *sp = P->ssp + (long long)r * ng;
        float s = 0.f;
        for (int c0 = 0; c0 < ng; c0 += 32 * 16) {
            float v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int c = c0 + lane + 32 * j;
                v[j] = c < ng ? sp[c] : 0.f;
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) s += v[j];
        }
        s = warp_sum(s);
        if (lane == 0) inv[r] = 1.0f / sqrtf(s / (float)P->d + P->eps);
    }
}

// Stage the slab [k0, k0 + kw) of all R rows: items are 4-element groups, U in flight per
// thread.  Normalised inputs are staged as x * g: the row's 1/rms scales the GEMM's output.
template <typename XT, int OP>
static __device__ __noinline__ void pg_stage_x(const Plan *__restrict__ P, const PdmRows &pr, int layer, int k0, int kw,
                                               unsigned char *xs, int pitch) {
    constexpr bool NORM = OP == OP_QKV || OP == OP_GATEUP;
    constexpr int U = NORM ? 8 : 16;
    const int R = pr.R, kw4 = kw >> 2, total = R * kw4, d = P->d;
    const float *g = OP == OP_QKV ? P->pl[layer].g1 : OP == OP_GATEUP ? P->pl[layer].g2 : nullptr;
    for (int b = threadIdx.x; b < total; b += U * PG_CONSUMERS) {
        float4 v[U], w[NORM ? U : 1];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = b + u * PG_CONSUMERS;
            if (i >= total) continue;
            const int r = i / kw4, k = k0 + 4 * (i - r * kw4);
            if (OP == OP_PROJ) {
                // anchor a of the row's slot (read whatever the depth; masked below)
                const int a = k / d, off = k - a * d;
                v[u] = *reinterpret_cast<const float4 *>(P->ANCH + ((long long)pr.slot[r] * P->nB + a) * d + off);
            } else if (NORM) {
                v[u] = *reinterpret_cast<const float4 *>(P->Xp + (long long)r * d + k);
                w[u] = *reinterpret_cast<const float4 *>(g + k);
            } else if (OP == OP_OPROJ) {
                v[u] = *reinterpret_cast<const float4 *>(P->ATTp + (long long)r * P->q_rows + k);
            } else {
                v[u] = *reinterpret_cast<const float4 *>(P->GUp + (long long)r * P->F + k);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = b + u * PG_CONSUMERS;
            if (i >= total) continue;
            const int r = i / kw4, kk = 4 * (i - r * kw4);
            float4 x = v[u];
            if (OP == OP_PROJ) {
                if (P->anchors[(k0 + kk) / d] > pr.depth[r]) x = make_float4(0.f, 0.f, 0.f, 0.f);
            } else if (NORM) {
                x = make_float4(x.x * w[u].x, x.y * w[u].y, x.z * w[u].z, x.w * w[u].w);
            }
            pg_store4<XT>(xs, pitch, r, kk, x);
        }
    }
}

// The global values that the epilogue of output (x row xr, weight row `row`, tile slot wr)
// reads, loaded ahead of it so that their latency overlaps the GEMM: QKV: the rotation's
// (cos, sin); projection, O, down: (residual, weight of the next normalisation).
template <typename T, int OP>
__device__ __forceinline__ float2 pg_prefetch(const Plan *__restrict__ P, const PdmRows &pr, int layer, int xr, int row,
                                              int wr, bool valid) {
    float2 r = make_float2(0.f, 0.f);
    if (!valid) return r;
    if (OP == OP_QKV) {
        if (row < P->q_rows + P->kv_rows) {
            const int pos = pr.pos0 + xr, hd = P->hd, half = hd >> 1, i = row % hd;
            r = P->rope[(long long)pos * half + (wr < 4 ? i : i - half)];
        }
    } else if (OP == OP_PROJ || OP == OP_OPROJ || OP == OP_DOWN) {
        if (OP != OP_PROJ) r.x = P->Xp[(long long)xr * P->d + row];
        if (sizeof(T) == 2) {
            // next normalisation: the next GEMM's, after the last layer the LM head's
            const float *gn = OP == OP_PROJ ? P->pl[0].g1 : OP == OP_OPROJ ? P->pl[layer].g2
                            : layer + 1 < P->Ls ? P->pl[layer + 1].g1 : P->pdm_gf;
            r.y = gn[row];
        }
    }
    return r;
}

// Finish output (x row xr, weight row `row`, tile slot wr) of group g with value v.  Called
// by whole warps of the reduction threads (tid < 128 MT), each thread owning the fixed
// (xr, wr) pair of the mma fragment layout; `valid` = the pair is a real output.  inv: the
// rows' 1/rms (QKV, gate/up: their x was staged unscaled); pre: pg_prefetch's values.
template <typename T, int OP>
__device__ __forceinline__ void pg_finish(const Plan *__restrict__ P, const PdmRows &pr, int layer, int g, int xr, int row,
                                          int wr, float v, bool valid, const float *inv, float2 pre) {
    if (OP == OP_QKV || OP == OP_GATEUP) {
        if (valid) v *= inv[xr];
    }
    if (OP == OP_QKV) {
        // rotary partner: slot wr ^ 4 of the same x row sits in lane ^ 2 (thread bit 3)
        const float partner = __shfl_xor_sync(0xffffffffu, v, 8);
        if (!valid) return;
        const int pos = pr.pos0 + xr;
        const long long cache = (long long)layer * P->kv_stride + (long long)pos * P->kv_rows;
        if (row < P->q_rows + P->kv_rows) {
            const bool first = wr < 4;
            const float2 cs = pre;
            const float a = first ? v : partner, b = first ? partner : v;
            const float y = first ? a * cs.x - b * cs.y : b * cs.x + a * cs.y;
            if (row < P->q_rows) P->QKVp[(long long)xr * P->qkv_rows + row] = y;
            else reinterpret_cast<KvT<T> *>(P->pkc)[cache + (row - P->q_rows)] = WTraits<KvT<T>>::store(y);
        } else {
            reinterpret_cast<KvT<T> *>(P->pvc)[cache + (row - P->q_rows - P->kv_rows)] = WTraits<KvT<T>>::store(v);
        }
    } else if (OP == OP_GATEUP) {
        // slots 0-3 hold gate rows u, slots 4-7 the up rows F + u, in lane ^ 2 (thread bit 3)
        const float up = __shfl_xor_sync(0xffffffffu, v, 8);
        if (valid && wr < 4) {
            const float h = silu_f(v) * up;
            if (sizeof(T) == 2) store_hilo(P->GUb, (long long)(P->n + 1) * P->F, (long long)xr * P->F + row, h);
            else P->GUp[(long long)xr * P->F + row] = h;
        }
    } else {
        float o = 0.f;
        if (valid) {
            o = OP == OP_PROJ ? v : pre.x + v;
            P->Xp[(long long)xr * P->d + row] = o;
            // bf16 input row of the next GEMM: x * g of its normalisation; after the last layer
            // the newest row is the LM head's second input row
            if (sizeof(T) == 2) {
                if (OP != OP_DOWN || layer + 1 < P->Ls)
                    store_hilo(P->Xb, (long long)(P->n + 1) * P->d, (long long)xr * P->d + row, o * pre.y);
                else if (xr == pr.R - 1) {
                    // the LM head's second input row in two bf16 parts: the value and the rest
                    const float xl = o * pre.y;
                    const __nv_bfloat16 hi = __float2bfloat16_rn(xl);
                    P->Xlm[P->d + row] = hi;
                    P->Xlm[3 * P->d + row] = __float2bfloat16_rn(xl - __bfloat162float(hi));
                }
            }
        }
        // sum of squares of the 8 rows of this group for x row xr (lanes differing in thread
        // bits 0, 2, 3 hold its 8 weight rows)
        float sq = o * o;
        sq += __shfl_xor_sync(0xffffffffu, sq, 1);
        sq += __shfl_xor_sync(0xffffffffu, sq, 4);
        sq += __shfl_xor_sync(0xffffffffu, sq, 8);
        if ((threadIdx.x & 13) == 0 && xr < pr.R) P->ssp[(long long)xr * (P->d / 8) + g] = sq;
    }
}

// Register-resident x: when one 16-row mma tile covers the rows, the whole K of the GEMM is
// one piece of a tile and each warp's K blocks are at most PG_XRB, every warp loads the A
// fragments of its blocks from the staged x once and keeps them in registers for the whole
// launch (the same K blocks meet every tile).
__host__ __device__ inline bool pg_xreg(int MT, int esz, int K, int ns) {
    return MT == 1 && esz == 2 && ns == 1 && K * esz <= PG_ROWB && K <= 8 * PG_XRB * PG_KB;
}

// ---- LM head on the same machinery (bf16, tied head): rows 0 and 1 of x are the final
// normalisation's x * g of the token leaving the last stage and of the draft module's
// newest row, left as bf16 by the target's last down projection and the draft's last down
// GEMM; their 1/rms scale the logits.

// 1/rms of the two rows, 0 for an absent row (no token leaves the last stage; no draft
// module): row 0 from the residual of the last stage's slot (warp 0, lane-strided loads in
// flight together, then the shuffle tree), row 1 from the draft's per-8-row sums of squares
// of its newest row (warp 1).
static __device__ __noinline__ void pg_lm_inv_rms(const Plan *__restrict__ P, const PdmRows &pr, float *inv) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, d = P->d;
    if (warp > 1) return;
    bool ok;
    float s = 0.f;
    if (warp == 0) {
        const DevState *st = P->st;
        const int n = P->n, es = ring(st->head, n - 1, n + 1);
        ok = st->valid[es] != 0;
        if (ok) {
            const float4 *x = reinterpret_cast<const float4 *>(P->X + (long long)es * d);
            const int n4 = d >> 2;
            for (int c0 = 0; c0 < n4; c0 += 32 * 16) {
                float4 v[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int c = c0 + lane + 32 * j;
                    v[j] = c < n4 ? x[c] : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    s = fmaf(v[j].x, v[j].x, s);
                    s = fmaf(v[j].y, v[j].y, s);
                    s = fmaf(v[j].z, v[j].z, s);
                    s = fmaf(v[j].w, v[j].w, s);
                }
            }
        }
    } else {
        const int r = pr.R - 1, ng = d / 8;
        ok = P->Ls > 0 && r >= 0;
        if (ok) {
            const float *sp = P->ssp + (long long)r * ng;
            for (int c0 = 0; c0 < ng; c0 += 32 * 16) {
                float v[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int c = c0 + lane + 32 * j;
                    v[j] = c < ng ? sp[c] : 0.f;
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) s += v[j];
            }
        }
    }
    s = warp_sum(s);
    if (lane == 0) inv[warp] = ok ? 1.0f / sqrtf(s / (float)d + P->eps) : 0.f;
}

// Argmax of the two logit rows (lowest id on ties): the CTA's candidates (held by the
// reduction threads of x rows 0 and 1, one per tile slot) are reduced in slot order, then
// the last CTA to finish merges the CTAs' results and leaves top / topval in the state.
// At T > 0 the same threads also carry their outputs' softmax statistics (running max of
// z/T and the sum of exp(z/T - max)): the CTA merges them in slot order, the last CTA merges
// the CTAs' in CTA order into the rows' normalisers, and draws the draft token from row 1 by
// inverse CDF (the smallest id whose running sum in id order exceeds u * total; CTAs hold
// consecutive id ranges, so the running sum is the CTA totals' prefix, then the crossing
// CTA's ids one warp-wide scan at a time).
static __device__ __noinline__ void pg_lm_argmax(const Plan *__restrict__ P, int xr, int wr, float bv, int bi, float sm,
                                                 float ss, int G8) {
    __shared__ float s_lv[2][PG_RG], s_sm[2][PG_RG], s_ss[2][PG_RG];
    __shared__ int s_li[2][PG_RG];
    __shared__ int s_last;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool stats = P->lm_stats != 0;
    if (tid < 128 && xr < 2) {
        s_lv[xr][wr] = bv;
        s_li[xr][wr] = bi;
        s_sm[xr][wr] = sm;
        s_ss[xr][wr] = ss;
    }
    named_sync(PG_BAR, PG_CONSUMERS);
    if (tid < 2) {
        float cv = -INFINITY;
        int ci = 0x7fffffff;
        for (int w = 0; w < PG_RG; ++w)
            if (s_lv[tid][w] > cv || (s_lv[tid][w] == cv && s_li[tid][w] < ci)) {
                cv = s_lv[tid][w];
                ci = s_li[tid][w];
            }
        P->lm_part[blockIdx.x * 4 + tid * 2] = cv;
        P->lm_part[blockIdx.x * 4 + tid * 2 + 1] = __int_as_float(ci);
        if (stats) {
            float m = -INFINITY;
            for (int w = 0; w < PG_RG; ++w) m = fmaxf(m, s_sm[tid][w]);
            float sum = 0.f;
            for (int w = 0; w < PG_RG; ++w)
                if (s_sm[tid][w] > -INFINITY) sum += s_ss[tid][w] * expf(s_sm[tid][w] - m);
            P->lm_stat[blockIdx.x * 4 + tid * 2] = m;
            P->lm_stat[blockIdx.x * 4 + tid * 2 + 1] = sum;
        }
    }
    __threadfence();
    named_sync(PG_BAR, PG_CONSUMERS);
    if (tid == 0) s_last = atomicAdd(P->lm_cnt, 1) == (int)gridDim.x - 1;
    named_sync(PG_BAR, PG_CONSUMERS);
    if (!s_last) return;
    __threadfence();
    const int nc = (int)gridDim.x;
    if (warp < 2) {
        const int row = warp;
        float cv = -INFINITY;
        int ci = 0x7fffffff;
        for (int c = lane; c < nc; c += 32) {
            const float v = __ldcg(P->lm_part + c * 4 + row * 2);
            const int id = __float_as_int(__ldcg(P->lm_part + c * 4 + row * 2 + 1));
            if (v > cv || (v == cv && id < ci)) {
                cv = v;
                ci = id;
            }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, cv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, ci, o);
            if (ov > cv || (ov == cv && oi < ci)) {
                cv = ov;
                ci = oi;
            }
        }
        if (lane == 0) {
            P->st->top[row] = ci;
            P->st->topval[row] = cv;
        }
        if (stats) {
            // the row's normaliser: max over the CTAs, then sum_c s_c e^{m_c - M} (lane-strided in
            // CTA order, then a fixed shuffle tree)
            float M = -INFINITY;
            for (int c = lane; c < nc; c += 32) M = fmaxf(M, __ldcg(P->lm_stat + c * 4 + row * 2));
            M = warp_max(M);
            float S = 0.f;
            for (int c = lane; c < nc; c += 32) {
                const float mc = __ldcg(P->lm_stat + c * 4 + row * 2);
                if (mc > -INFINITY) S += __ldcg(P->lm_stat + c * 4 + row * 2 + 1) * expf(mc - M);
            }
            S = warp_sum(S);
            if (lane == 0) {
                P->st->lmM[row] = M;
                P->st->lmS[row] = S;
            }
            if (row == 1 && !P->forced) {
                // the draft token: u0 = the step's purpose-0 uniform
                const uint32_t t = (uint32_t)(P->st->t + 1);
                const float u0 = (float)(philox_word0(t, 0u, P->seed_lo, P->seed_hi) >> 8) * (1.0f / 16777216.0f);
                const float target = u0 * S;
                // the crossing CTA: running sum of the CTA totals in CTA order, 32 at a time
                float before = 0.f;
                int cstar = nc - 1;
                for (int c0 = 0; c0 < nc; c0 += 32) {
                    const int c = c0 + lane;
                    const float mc = c < nc ? __ldcg(P->lm_stat + c * 4 + 2) : -INFINITY;
                    const float w = mc > -INFINITY ? __ldcg(P->lm_stat + c * 4 + 3) * expf(mc - M) : 0.f;
                    float inc = w;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const float y = __shfl_up_sync(0xffffffffu, inc, o);
                        if (lane >= o) inc += y;
                    }
                    const unsigned hit = __ballot_sync(0xffffffffu, c < nc && w > 0.f && before + inc > target);
                    if (hit) {
                        const int l = __ffs(hit) - 1;
                        const float ex = __shfl_sync(0xffffffffu, inc - w, l);
                        before += ex;
                        cstar = c0 + l;
                        break;
                    }
                    before += __shfl_sync(0xffffffffu, inc, 31);
                }
                // the crossing CTA's ids, in id order
                const float invT = 1.0f / P->temperature;
                const float *z = P->logits + P->V;
                // CTA c holds tile groups [G8 c / nc, G8 (c + 1) / nc) of 8 ids each
                const int i0 = 8 * (int)((long long)G8 * cstar / nc);
                const int i1 = min(P->V, 8 * (int)((long long)G8 * (cstar + 1) / nc));
                int pick = -1, lastnz = -1;
                for (int b0 = i0; b0 < i1 && pick < 0; b0 += 32) {
                    const int i = b0 + lane;
                    const float w = i < i1 ? expf(z[i] * invT - M) : 0.f;
                    float inc = w;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const float y = __shfl_up_sync(0xffffffffu, inc, o);
                        if (lane >= o) inc += y;
                    }
                    const unsigned hit = __ballot_sync(0xffffffffu, i < i1 && w > 0.f && before + inc > target);
                    const unsigned nz = __ballot_sync(0xffffffffu, i < i1 && w > 0.f);
                    if (nz) lastnz = b0 + 31 - __clz(nz);
                    if (hit) pick = b0 + __ffs(hit) - 1;
                    before += __shfl_sync(0xffffffffu, inc, 31);
                }
                if (lane == 0) P->st->samp = pick >= 0 ? pick : (lastnz >= 0 ? lastnz : min(i0, P->V - 1));
            }
        }
    }
    if (tid == 0) *P->lm_cnt = 0;
}

// One CTA's share of a draft GEMM: CTA p of m_pdm (row block p / ns, K slab p % ns).
// smem: the dynamic shared memory; full/empty: PG_MAXNS mbarriers each, initialised (full
// count 1, empty count 8) and fenced by the caller, like xbar (count 1: the bf16 x rows'
// copies); s_inv: MAXS floats.  Called by all
// PG_THREADS threads (warp 8 is the producer); returns when the CTA's work is done.
template <typename T, int OP, int MT>
__device__ void pdm_gemm_cta(const Plan *__restrict__ P, const PdmRows &pr, int layer, int p, int m_pdm,
                             unsigned char *smem, uint64_t *full, uint64_t *empty, uint64_t *xbar, float *s_inv,
                             int *s_flag) {
    constexpr int ESZ = sizeof(T);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, tid = threadIdx.x;
    const int ns = P->pdm_ns[OP], kx = P->pdm_kx[OP];
    const int N = pg_N<OP>(*P), K = pg_K<OP>(*P), G8 = N / 8;
    const int nb = m_pdm / ns, b = p / ns, sl = p - (p / ns) * ns;
    if (b >= nb || (OP != OP_LM && pr.R < 1)) return;
    // LM head: rows 0, 1 = the token leaving the last stage and the draft module's newest row
    // (bf16 of x * g_final), rows 2, 3 = bf16 of what rows 0, 1 left out of x * g_final; the
    // products of rows r and r + 2 are added, so the head sees x at about 16 mantissa bits
    const int R = OP == OP_LM ? 4 : pr.R;
    const int k0 = sl * kx, kw = min(kx, K - k0);
    const int gb0 = (int)((long long)G8 * b / nb), gb1 = (int)((long long)G8 * (b + 1) / nb);
    const int nch = pg_nch(kw, ESZ), KC = pg_kc(kw, ESZ);
    const int xpitch = pg_pitch(kx, ESZ);
    const int rowb = pg_pitch(KC, ESZ), stage_bytes = PG_RG * rowb;
    const bool xreg = pg_xreg(MT, ESZ, K, ns);
    // bf16 weights: the inputs are bf16 rows in global memory already, copied whole into x by
    // bulk copies (the projection's per anchor, masked ones zeroed instead); the
    // register-resident fragments are then read from there
    constexpr bool BULK = ESZ == 2;
    // x rows in shared memory: rows 0..n the hi parts, rows n+1..2n+1 the lo parts (bf16, but
    // not the LM head, whose four rows carry both parts of its two rows already)
    constexpr bool HILO = ESZ == 2 && pg_hilo<OP>();
    const int xrows = OP == OP_LM ? 4 : (HILO ? 2 : 1) * (P->n + 1);
    const int xbytes = pg_xbytes(xrows, kx, ESZ);
    unsigned char *xs = smem;
    unsigned char *xlo = xs + (P->n + 1) * xpitch;   // lo rows (HILO)
    float4 *red = reinterpret_cast<float4 *>(smem + xbytes);
    unsigned char *stages = smem + xbytes + pg_redbytes(MT);
    const int NS = min(PG_MAXNS, (PG_SMEM - xbytes - pg_redbytes(MT)) / stage_bytes);
    const PgRows<T, OP> wrows = pg_rows<T, OP>(P, layer);

    if (warp == PG_CONSUMERS / 32) {
        // ------------------------------ producer ----------------------------------------
        if (lane == 0) {
            uint32_t tile = 0;
            for (int g = gb0; g < gb1; ++g) {
                const T *rp[PG_RG];
#pragma unroll
                for (int q = 0; q < PG_RG; ++q) rp[q] = wrows.ptr(wrows.row_of(g, q)) + k0;
                for (int c = 0; c < nch; ++c) {
                    const int kc0 = c * KC, len = min(KC, kw - kc0);
                    const int sidx = tile % NS;
                    const uint32_t u = tile / NS;
                    if (!mbar_wait(&empty[sidx], (u & 1) ^ 1)) P->st->error = ERR_TIMEOUT;
                    const uint32_t bytes = (uint32_t)len * ESZ;
                    mbar_expect_tx(&full[sidx], bytes * PG_RG);
#pragma unroll
                    for (int q = 0; q < PG_RG; ++q) bulk_g2s(stages + sidx * stage_bytes + q * rowb, rp[q] + kc0, bytes, &full[sidx]);
                    ++tile;
                }
            }
        }
        return;
    }

    // ------------------------------ consumers -------------------------------------------
    pdl_wait();   // x, its statistics and the counters belong to the preceding launch
    pdl_trigger();
    if constexpr (BULK && OP == OP_PROJ) {
        // row r, anchor a: the piece [max(k0, a d), min(k0 + kw, (a + 1) d)) of the slab
        const int d = P->d, a0 = k0 / d, a1 = (k0 + kw - 1) / d;
        const long long alo = (long long)(P->n + 1) * P->nB * d;   // the anchors' lo parts
        if (tid == 0) {
            uint32_t tot = 0;
            for (int r = 0; r < R; ++r)
                for (int a = a0; a <= a1; ++a)
                    if (P->anchors[a] <= pr.depth[r]) tot += (uint32_t)(min(k0 + kw, (a + 1) * d) - max(k0, a * d)) * 4;
            fence_proxy_async();
            mbar_expect_tx(xbar, tot);
            for (int r = 0; r < R; ++r)
                for (int a = a0; a <= a1; ++a) {
                    if (P->anchors[a] > pr.depth[r]) continue;
                    const int ka = max(k0, a * d), kb = min(k0 + kw, (a + 1) * d);
                    const __nv_bfloat16 *src = P->ANCHb + ((long long)pr.slot[r] * P->nB + a) * d + (ka - a * d);
                    bulk_g2s(xs + r * xpitch + (ka - k0) * 2, src, (uint32_t)(kb - ka) * 2, xbar);
                    bulk_g2s(xlo + r * xpitch + (ka - k0) * 2, src + alo, (uint32_t)(kb - ka) * 2, xbar);
                }
        }
        // anchors deeper than the row's token enter as zeros (both parts)
        for (int r = 0; r < R; ++r)
            for (int a = a0; a <= a1; ++a) {
                if (P->anchors[a] <= pr.depth[r]) continue;
                const int ka = max(k0, a * d), kb = min(k0 + kw, (a + 1) * d);
                for (int e = ka + 8 * tid; e < kb; e += 8 * PG_CONSUMERS) {
                    *reinterpret_cast<uint4 *>(xs + r * xpitch + (e - k0) * 2) = make_uint4(0u, 0u, 0u, 0u);
                    *reinterpret_cast<uint4 *>(xlo + r * xpitch + (e - k0) * 2) = make_uint4(0u, 0u, 0u, 0u);
                }
            }
    } else if constexpr (BULK) {
        if (tid == 0) {
            const __nv_bfloat16 *src = OP == OP_OPROJ ? P->ATTb : OP == OP_DOWN ? P->GUb : OP == OP_LM ? P->Xlm : P->Xb;
            const long long lo = (long long)(P->n + 1) * K;   // lo parts (if any) follow the hi parts
            const uint32_t rb = (uint32_t)kw * 2;
            fence_proxy_async();
            mbar_expect_tx(xbar, rb * R * (HILO ? 2 : 1));
            for (int r = 0; r < R; ++r) {
                bulk_g2s(xs + r * xpitch, src + (long long)r * K + k0, rb, xbar);
                if (HILO) bulk_g2s(xlo + r * xpitch, src + lo + (long long)r * K + k0, rb, xbar);
            }
        }
    } else if (!xreg) {
        pg_stage_x<T, OP>(P, pr, layer, k0, kw, xs, xpitch);
    }
    // the rows' 1/rms (read by the epilogue, after the first group's barrier at the latest)
    if (OP == OP_QKV || OP == OP_GATEUP) pg_row_inv_rms(P, R, s_inv);
    if (OP == OP_LM) pg_lm_inv_rms(P, pr, s_inv);
    if constexpr (BULK) {
        if (!mbar_wait(xbar, 0)) P->st->error = ERR_TIMEOUT;
        if (OP == OP_PROJ) named_sync(PG_BAR, PG_CONSUMERS);   // the zeroed pieces
    } else if (!xreg) {
        named_sync(PG_BAR, PG_CONSUMERS);
    }
    // register-resident x (bf16, one mma tile): lane (gq, tq) of warp w holds rows gq and gq + 8,
    // elements 8tq..8tq+7 of blocks w, w + 8, ... of the GEMM's K
    uint4 xf[PG_XRB][2];
    if constexpr (ESZ == 2 && MT == 1) {
        if (xreg) {
            const int gq = lane >> 2, tq = lane & 3, nblk = kw / PG_KB;
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int j = 0; j < PG_XRB; ++j) {
                const int bb = warp + 8 * j, kl = bb * PG_KB + 8 * tq;
                xf[j][0] = bb < nblk && gq < R ? lds128(xs + gq * xpitch + kl * 2) : z;
                xf[j][1] = bb < nblk && gq + 8 < R ? lds128(xs + (gq + 8) * xpitch + kl * 2) : z;
            }
        }
    }

    // reduction thread t (< 128 MT) owns x row xr_t and tile slot wr_t of every group
    const int rm = tid >> 7, rl = (tid >> 2) & 31, rreg = tid & 3;
    const int xr_t = rm * 16 + (rreg >> 1) * 8 + (rl >> 2), wr_t = (rl & 3) * 2 + (rreg & 1);
    float *part = P->pdm_part;   // [ns][n+1][N] slab partials
    const int gq = lane >> 2, tq = lane & 3;
    uint32_t tile = 0;
    int buf = 0;
    // LM head: this thread's argmax candidate and the draft row's logits for sampling
    float lbv = -INFINITY, lsm = -INFINITY, lss = 0.f;   // argmax; softmax statistics at T > 0
    int lbi = 0x7fffffff;
    float *dl = nullptr;
    if (OP == OP_LM && P->temperature > 0.f) dl = P->dlogits + (long long)ring(P->st->head + 1, 0, P->n + 1) * P->V;
    for (int g = gb0; g < gb1; ++g) {
        float2 pre = make_float2(0.f, 0.f);
        if (ns == 1 && tid < 128 * MT) pre = pg_prefetch<T, OP>(P, pr, layer, xr_t, wrows.row_of(g, wr_t), wr_t, xr_t < R);
        // bf16: acc[4m..4m+3] is the m-th 16x8 mma accumulator fragment; fp32: acc[j] is the
        // (x row (lane >> 3) + 4j, tile slot lane & 7) product
        float acc[4 * MT];
#pragma unroll
        for (int j = 0; j < 4 * MT; ++j) acc[j] = 0.f;
        for (int c = 0; c < nch; ++c) {
            const int kc0 = c * KC, len = min(KC, kw - kc0), nblk = len / PG_KB;
            const int sidx = tile % NS;
            const uint32_t u = tile / NS;
            if (!mbar_wait(&full[sidx], u & 1)) P->st->error = ERR_TIMEOUT;
            const unsigned char *tb = stages + sidx * stage_bytes;
            bool done_xreg = false;
            if constexpr (ESZ == 2 && MT == 1) {
                if (xreg) {
                    // one piece per tile (nch == 1): block bb = warp + 8j uses the j-th registers
                    // for the hi parts; lo parts, where the GEMM has them, come from shared memory
                    const unsigned char *wp = tb + gq * rowb + tq * 16;
                    const unsigned char *lp = xlo + gq * xpitch + tq * 16;
                    const bool l0 = gq < R, l1 = gq + 8 < R;
                    float acc2[4] = {0.f, 0.f, 0.f, 0.f};
                    float(&f)[4] = *reinterpret_cast<float(*)[4]>(&acc[0]);
#pragma unroll
                    for (int j = 0; j < PG_XRB; ++j) {
                        const int bb = warp + 8 * j;
                        if (bb < nblk) {
                            const uint4 w = lds128(wp + bb * 64);
                            mma_bf16(f, xf[j][0].x, xf[j][1].x, xf[j][0].y, xf[j][1].y, w.x, w.y);
                            mma_bf16(acc2, xf[j][0].z, xf[j][1].z, xf[j][0].w, xf[j][1].w, w.z, w.w);
                            if (HILO) {
                                const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                                const uint4 la = l0 ? lds128(lp + bb * 64) : z;
                                const uint4 lb = l1 ? lds128(lp + 8 * xpitch + bb * 64) : z;
                                mma_bf16(f, la.x, lb.x, la.y, lb.y, w.x, w.y);
                                mma_bf16(acc2, la.z, lb.z, la.w, lb.w, w.z, w.w);
                            }
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[j] += acc2[j];
                    done_xreg = true;
                }
            }
            if (done_xreg) {
            } else if constexpr (ESZ == 2) {
                // lane (gq, tq): tile slot gq, x rows gq and gq + 8 (+16 m), elements 8tq..8tq+7 of
                // each 32-block; the two mma steps take elements {8tq..8tq+3} and {8tq+4..8tq+7}
                // and go to two accumulator chains (added at the end of the piece)
                const unsigned char *wp = tb + gq * rowb + tq * 16;
                const unsigned char *xp = xs + gq * xpitch + kc0 * 2 + tq * 16;
                const unsigned char *xq = xlo + gq * xpitch + kc0 * 2 + tq * 16;
                bool xv[MT][2];
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    xv[m][0] = m * 16 + gq < R;
                    xv[m][1] = m * 16 + 8 + gq < R;
                }
                float acc2[4 * MT];
#pragma unroll
                for (int j = 0; j < 4 * MT; ++j) acc2[j] = 0.f;
                for (int bb = warp; bb < nblk; bb += PG_CONSUMERS / 32) {
                    const uint4 w = lds128(wp + bb * 64);
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                        const uint4 xa = xv[m][0] ? lds128(xp + (m * 16) * xpitch + bb * 64) : z;
                        const uint4 xb = xv[m][1] ? lds128(xp + (m * 16 + 8) * xpitch + bb * 64) : z;
                        float(&f)[4] = *reinterpret_cast<float(*)[4]>(&acc[4 * m]);
                        float(&f2)[4] = *reinterpret_cast<float(*)[4]>(&acc2[4 * m]);
                        mma_bf16(f, xa.x, xb.x, xa.y, xb.y, w.x, w.y);
                        mma_bf16(f2, xa.z, xb.z, xa.w, xb.w, w.z, w.w);
                        if (HILO) {
                            const uint4 la = xv[m][0] ? lds128(xq + (m * 16) * xpitch + bb * 64) : z;
                            const uint4 lb = xv[m][1] ? lds128(xq + (m * 16 + 8) * xpitch + bb * 64) : z;
                            mma_bf16(f, la.x, lb.x, la.y, lb.y, w.x, w.y);
                            mma_bf16(f2, la.z, lb.z, la.w, lb.w, w.z, w.w);
                        }
                    }
                }
#pragma unroll
                for (int j = 0; j < 4 * MT; ++j) acc[j] += acc2[j];
            } else {
                // fp32 weights: plain FMAs in element order
                const int wrow = lane & 7, xq = lane >> 3;
                const float *wp = reinterpret_cast<const float *>(tb + wrow * rowb);
                for (int bb = warp; bb < nblk; bb += PG_CONSUMERS / 32) {
                    for (int e = 0; e < PG_KB; ++e) {
                        const int k = bb * PG_KB + e;
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
        // ---- partial products of all warps in the fragment layout [buf][warp][m][lane] x 4:
        // float (m, lane, reg) = (x row 16m + 8(reg >> 1) + lane / 4, slot 2(lane % 4) + reg % 2)
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
            const float *rf = reinterpret_cast<const float *>(red);
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < PG_CONSUMERS / 32; ++w) s += rf[(((buf * (PG_CONSUMERS / 32) + w) * MT + rm) * 32 + rl) * 4 + rreg];
            const int row = wrows.row_of(g, wr_t);
            if constexpr (OP == OP_LM) {
                if (xr_t < 2) {
                    // x row xr_t + 2 (the remainder part) sits 8 fragment lanes further
                    float lo = 0.f;
#pragma unroll
                    for (int w = 0; w < PG_CONSUMERS / 32; ++w)
                        lo += rf[(((buf * (PG_CONSUMERS / 32) + w) * MT + rm) * 32 + rl + 8) * 4 + rreg];
                    const float z = (s + lo) * s_inv[xr_t];
                    P->logits[(long long)xr_t * N + row] = z;
                    if (xr_t == 1 && dl) dl[row] = z;
                    if (z > lbv || (z == lbv && row < lbi)) {
                        lbv = z;
                        lbi = row;
                    }
                    if (P->lm_stats) {
                        const float v = z / P->temperature;
                        if (v > lsm) {
                            lss = lss * expf(lsm - v) + 1.f;
                            lsm = v;
                        } else {
                            lss += expf(v - lsm);
                        }
                    }
                }
            } else if (ns == 1) {
                pg_finish<T, OP>(P, pr, layer, g, xr_t, row, wr_t, s, xr_t < R, s_inv, pre);
            } else if (xr_t < R) {
                part[((long long)sl * (P->n + 1) + xr_t) * N + row] = s;
            }
        }
        buf ^= 1;
    }
    if constexpr (OP == OP_LM) {
        pg_lm_argmax(P, xr_t, wr_t, lbv, lbi, lsm, lss, G8);
        return;
    }
    if (ns == 1) return;

    // ---- K slabs: the last CTA of the row block adds the slab partials in slab order
    __threadfence();
    named_sync(PG_BAR, PG_CONSUMERS);
    if (tid == 0) *s_flag = atomicAdd(P->pdm_cnt + b, 1) == ns - 1;
    named_sync(PG_BAR, PG_CONSUMERS);
    if (!*s_flag) return;
    __threadfence();
    // all consumer threads: 256 / (128 MT) groups per pass, PG_FIN passes' slab loads in flight
    // together; thread t keeps the fixed (x row, slot) pair of the fragment layout
    {
        constexpr int GPP = 2 / MT;          // groups per pass
        constexpr int PG_FIN = 4;            // passes per batch
        const int gsub = tid / (128 * MT), t = tid - gsub * (128 * MT);
        const int xr = (t >> 7) * 16 + ((t & 3) >> 1) * 8 + ((t >> 2) & 31) / 4, wr = (((t >> 2) & 31) & 3) * 2 + (t & 1);
        for (int g0 = gb0; g0 < gb1; g0 += GPP * PG_FIN) {
            float sum[PG_FIN];
            float2 pre[PG_FIN];
#pragma unroll
            for (int f = 0; f < PG_FIN; ++f) {
                sum[f] = 0.f;
                const int g = g0 + f * GPP + gsub;
                pre[f] = pg_prefetch<T, OP>(P, pr, layer, xr, wrows.row_of(min(g, gb1 - 1), wr), wr, g < gb1 && xr < R);
            }
            for (int s0 = 0; s0 < ns; s0 += 4) {
                float v[PG_FIN][4];
#pragma unroll
                for (int f = 0; f < PG_FIN; ++f) {
                    const int g = g0 + f * GPP + gsub;
                    const int row = wrows.row_of(min(g, gb1 - 1), wr);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        v[f][q] = (g < gb1 && xr < R && s0 + q < ns)
                                      ? __ldcg(part + ((long long)(s0 + q) * (P->n + 1) + xr) * N + row) : 0.f;
                }
#pragma unroll
                for (int f = 0; f < PG_FIN; ++f)
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (s0 + q < ns) sum[f] += v[f][q];
            }
#pragma unroll
            for (int f = 0; f < PG_FIN; ++f) {
                const int g = g0 + f * GPP + gsub;
                // warp-uniform: the 32 threads of a warp share gsub, hence g
                if (g < gb1) pg_finish<T, OP>(P, pr, layer, g, xr, wrows.row_of(g, wr), wr, sum[f], xr < R, s_inv, pre[f]);
            }
        }
    }
    if (tid == 0) P->pdm_cnt[b] = 0;
}

}  // namespace spd
