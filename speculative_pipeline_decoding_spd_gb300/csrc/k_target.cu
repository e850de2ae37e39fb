// Target-model kernels of one pipeline step: the grouped per-stage GEMVs and the
// batched LM head.
//
// Speculative pipeline decoding (abstract; machine review "The reading"): the target is
// cut into n stages and the n in-flight tokens advance through their own stage in the
// same step.  Round j of a step runs layer b_s + j of every occupied stage s; each
// stage multiplies its own weight matrix by its own token's vector (N = 1 GEMV), so a
// round is a grouped GEMV over n different weight blocks.  The whole round's rows
// (stages x output rows) are spread evenly over all CTAs, so a partly filled pipeline
// (after a flush) still streams its weights with the full GPU.
//
// Per output row the arithmetic is fixed (each lane accumulates its 16-byte pieces in
// order, warp shuffle tree, then the 8 warp partials in order), so a token's result
// does not depend on which other stages run in the same step: the pipeline produces
// bit-identical hidden states to a one-token-at-a-time decode.
#include "common.cuh"

namespace spd {

enum { EPI_QKV = 0, EPI_OPROJ = 1, EPI_GATEUP = 2, EPI_DOWN = 3 };

constexpr int RG = 8;   // output rows per CTA group (gate/up: 4 pairs)
constexpr int UB = 2;   // 512-byte blocks per warp per batch

struct StageList {
    int m;
    int stage[MAXS], slot[MAXS], layer[MAXS];
};

// Occupied stages that have a layer at this round.
__device__ void build_stage_list(const Plan *__restrict__ P, int round, StageList &L) {
    const DevState *st = P->st;
    const int n = P->n, ns = n + 1, head = st->head;
    int m = 0;
    for (int s = 0; s < n; ++s) {
        const int slot = ring(head, s, ns);
        if (!st->valid[slot]) continue;
        const int layer = P->b[s] + round;
        if (layer >= P->b[s + 1]) continue;
        L.stage[m] = s;
        L.slot[m] = slot;
        L.layer[m] = layer;
        ++m;
    }
    L.m = m;
}

template <typename T, int EPI>
__device__ __forceinline__ const T *row_ptr(const Plan *__restrict__ P, const LayerW &w, int r, int K) {
    if (EPI == EPI_QKV) {
        if (r < P->q_rows) return reinterpret_cast<const T *>(w.wq) + (long long)r * K;
        r -= P->q_rows;
        if (r < P->kv_rows) return reinterpret_cast<const T *>(w.wk) + (long long)r * K;
        return reinterpret_cast<const T *>(w.wv) + (long long)(r - P->kv_rows) * K;
    } else if (EPI == EPI_OPROJ) {
        return reinterpret_cast<const T *>(w.wo) + (long long)r * K;
    } else if (EPI == EPI_DOWN) {
        return reinterpret_cast<const T *>(w.wd) + (long long)r * K;
    }
    return nullptr;
}

template <typename T, int EPI>
__global__ void __launch_bounds__(GEMV_THREADS, 2) k_target_gemv(const Plan *__restrict__ P, int round) {
    extern __shared__ __align__(16) float xs[];
    __shared__ StageList SL;
    __shared__ float red[GEMV_WARPS * RG + 33];
    __shared__ int s_done;
    if (threadIdx.x == 0) {
        s_done = P->st->done;
        build_stage_list(P, round, SL);
    }
    __syncthreads();
    if (s_done || SL.m == 0) return;

    constexpr int VEC = WTraits<T>::VEC;
    const int d = P->d;
    const int N = EPI == EPI_QKV ? P->qkv_rows : (EPI == EPI_GATEUP ? P->F : d);
    const int K = (EPI == EPI_QKV || EPI == EPI_GATEUP) ? d : (EPI == EPI_OPROJ ? P->q_rows : P->F);
    const int nvec = K / VEC;
    const int nblk = (nvec + 31) / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    const long long total = (long long)SL.m * N;
    const long long lo = total * blockIdx.x / gridDim.x;
    const long long hi = total * (blockIdx.x + 1) / gridDim.x;

    long long r = lo;
    while (r < hi) {
        const int i = (int)(r / N);
        const int r0 = (int)(r - (long long)i * N);
        const int r1 = (int)min((long long)N, hi - (long long)i * N);
        const int s = SL.stage[i], slot = SL.slot[i], layer = SL.layer[i];
        const LayerW &w = P->tl[layer];
        // ---- stage x for this stage
        if (EPI == EPI_QKV)
            stage_norm(P->X + (long long)slot * d, w.g1, d, P->eps, xs, red);
        else if (EPI == EPI_GATEUP)
            stage_norm(P->X + (long long)slot * d, w.g2, d, P->eps, xs, red);
        else if (EPI == EPI_OPROJ)
            stage_f4(P->ATT + (long long)s * P->q_rows, xs, K);
        else
            stage_f4(P->U + (long long)s * P->F, xs, K);
        __syncthreads();

        constexpr int GR = EPI == EPI_GATEUP ? RG / 2 : RG;   // output units per group
        for (int g0 = r0; g0 < r1; g0 += GR) {
            const T *wrow[RG];
            bool rv[RG];
#pragma unroll
            for (int q = 0; q < RG; ++q) {
                if (EPI == EPI_GATEUP) {
                    const int u = g0 + (q % GR);
                    rv[q] = u < r1;
                    const void *base = q < GR ? w.wg : w.wu;
                    wrow[q] = reinterpret_cast<const T *>(base) + (long long)(rv[q] ? u : g0) * K;
                } else {
                    const int rr = g0 + q;
                    rv[q] = rr < r1;
                    wrow[q] = row_ptr<T, EPI>(P, w, rv[q] ? rr : g0, K);
                }
            }
            float acc[RG];
#pragma unroll
            for (int q = 0; q < RG; ++q) acc[q] = 0.f;
            for (int b0 = warp; b0 < nblk; b0 += GEMV_WARPS * UB) {
                uint4 v[UB][RG];
#pragma unroll
                for (int u = 0; u < UB; ++u) {
                    const int vi = (b0 + u * GEMV_WARPS) * 32 + lane;
                    const bool ok = (b0 + u * GEMV_WARPS) < nblk && vi < nvec;
#pragma unroll
                    for (int q = 0; q < RG; ++q) {
                        if (ok && rv[q])
                            v[u][q] = ld_stream(wrow[q] + (long long)vi * VEC);
                        else
                            v[u][q] = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
#pragma unroll
                for (int u = 0; u < UB; ++u) {
                    const int vi = (b0 + u * GEMV_WARPS) * 32 + lane;
                    const bool ok = (b0 + u * GEMV_WARPS) < nblk && vi < nvec;
                    if (ok) {
                        const float *xv = xs + (long long)vi * VEC;
#pragma unroll
                        for (int q = 0; q < RG; ++q) acc[q] = dot16(v[u][q], xv, acc[q], T());
                    }
                }
            }
#pragma unroll
            for (int q = 0; q < RG; ++q) {
                const float t = warp_sum(acc[q]);
                if (lane == 0) red[warp * RG + q] = t;
            }
            __syncthreads();
            if (threadIdx.x < GR) {
                const int q = threadIdx.x;
                float sum = 0.f;
#pragma unroll
                for (int ww = 0; ww < GEMV_WARPS; ++ww) sum += red[ww * RG + q];
                const int rr = g0 + q;
                if (rr < r1) {
                    if (EPI == EPI_QKV) {
                        P->QKV[(long long)s * P->qkv_rows + rr] = sum;
                    } else if (EPI == EPI_OPROJ) {
                        P->X[(long long)slot * d + rr] += sum;
                    } else if (EPI == EPI_GATEUP) {
                        float up = 0.f;
#pragma unroll
                        for (int ww = 0; ww < GEMV_WARPS; ++ww) up += red[ww * RG + GR + q];
                        P->U[(long long)s * P->F + rr] = silu_f(sum) * up;
                    } else {
                        float *xp = P->X + (long long)slot * d + rr;
                        const float xn = *xp + sum;
                        *xp = xn;
                        const int a = P->aidx[layer + 1];
                        if (a >= 0) P->ANCH[((long long)slot * P->nB + a) * d + rr] = xn;
                    }
                }
            }
            __syncthreads();
        }
        r = (long long)(i + 1) * N;
    }
}

// ---------------------------------------------------------------------------------
// LM head for {target exit row, draft newest row}: logits = W_lm (rms(h) * g), the
// argmax with the lowest id on ties.  Tied heads stream W_lm once for both rows.
template <typename T, bool TIED>
__global__ void __launch_bounds__(GEMV_THREADS, 2) k_lm_head(const Plan *__restrict__ P) {
    extern __shared__ __align__(16) float xs[];   // [2][d]
    __shared__ float red[GEMV_WARPS * RG * 2 + 33];
    __shared__ int s_rows[2], s_done, s_last;
    __shared__ float s_bv[2][GEMV_THREADS / 32];
    __shared__ int s_bi[2][GEMV_THREADS / 32];
    const DevState *st = P->st;
    const int d = P->d, V = P->V, n = P->n, ns = n + 1;
    if (threadIdx.x == 0) {
        s_done = st->done;
        const int head = st->head;
        s_rows[0] = st->valid[ring(head, n - 1, ns)] ? ring(head, n - 1, ns) : -1;   // exit slot
        int R = st->pending ? 1 : 0;
        for (int s = 0; s < n; ++s) R += st->valid[ring(head, s, ns)] ? 1 : 0;
        s_rows[1] = R - 1;                                                          // newest draft row
    }
    __syncthreads();
    if (s_done) return;
    float *red2 = red + GEMV_WARPS * RG * 2;
    if (s_rows[0] >= 0)
        stage_norm(P->X + (long long)s_rows[0] * d, P->gf, d, P->eps, xs, red2);
    else
        for (int k = threadIdx.x; k < d; k += blockDim.x) xs[k] = 0.f;
    __syncthreads();
    if (P->Ls > 0)
        stage_norm(P->Xp + (long long)s_rows[1] * d, P->pdm_gf, d, P->eps, xs + d, red2);
    else
        for (int k = threadIdx.x; k < d; k += blockDim.x) xs[d + k] = 0.f;
    __syncthreads();

    constexpr int VEC = WTraits<T>::VEC;
    const int nvec = d / VEC, nblk = (nvec + 31) / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr bool tied = TIED;
    const T *W0 = reinterpret_cast<const T *>(P->lm_head);
    const T *W1 = reinterpret_cast<const T *>(P->pdm_lm_head);
    const int lo = (int)((long long)V * blockIdx.x / gridDim.x);
    const int hi = (int)((long long)V * (blockIdx.x + 1) / gridDim.x);
    float bv0 = -INFINITY, bv1 = -INFINITY;
    int bi0 = 0x7fffffff, bi1 = 0x7fffffff;
    const int newslot = ring(st->head + 1, 0, ns);
    float *dl = P->temperature > 0.f ? P->dlogits + (long long)newslot * V : nullptr;
    for (int g0 = lo; g0 < hi; g0 += RG) {
        float a0[RG], a1[RG];
#pragma unroll
        for (int q = 0; q < RG; ++q) a0[q] = a1[q] = 0.f;
        for (int b0 = warp; b0 < nblk; b0 += GEMV_WARPS * UB) {
            uint4 v[UB][RG], v1[TIED ? 1 : UB][TIED ? 1 : RG];
#pragma unroll
            for (int u = 0; u < UB; ++u) {
                const int vi = (b0 + u * GEMV_WARPS) * 32 + lane;
                const bool ok = (b0 + u * GEMV_WARPS) < nblk && vi < nvec;
#pragma unroll
                for (int q = 0; q < RG; ++q) {
                    const bool rv = ok && (g0 + q < hi);
                    v[u][q] = rv ? ld_stream(W0 + (long long)(g0 + q) * d + (long long)vi * VEC) : make_uint4(0, 0, 0, 0);
                    if constexpr (!TIED)
                        v1[u][q] = rv ? ld_stream(W1 + (long long)(g0 + q) * d + (long long)vi * VEC) : make_uint4(0, 0, 0, 0);
                }
            }
#pragma unroll
            for (int u = 0; u < UB; ++u) {
                const int vi = (b0 + u * GEMV_WARPS) * 32 + lane;
                const bool ok = (b0 + u * GEMV_WARPS) < nblk && vi < nvec;
                if (ok) {
                    const float *x0 = xs + (long long)vi * VEC;
                    const float *x1 = xs + d + (long long)vi * VEC;
#pragma unroll
                    for (int q = 0; q < RG; ++q) {
                        a0[q] = dot16(v[u][q], x0, a0[q], T());
                        if constexpr (TIED)
                            a1[q] = dot16(v[u][q], x1, a1[q], T());
                        else
                            a1[q] = dot16(v1[u][q], x1, a1[q], T());
                    }
                }
            }
        }
#pragma unroll
        for (int q = 0; q < RG; ++q) {
            const float t0 = warp_sum(a0[q]);
            const float t1 = warp_sum(a1[q]);
            if (lane == 0) {
                red[(warp * RG + q) * 2] = t0;
                red[(warp * RG + q) * 2 + 1] = t1;
            }
        }
        __syncthreads();
        if (threadIdx.x < 2 * RG) {
            const int q = threadIdx.x >> 1, row = threadIdx.x & 1;
            float sum = 0.f;
#pragma unroll
            for (int ww = 0; ww < GEMV_WARPS; ++ww) sum += red[(ww * RG + q) * 2 + row];
            const int v = g0 + q;
            if (v < hi) {
                P->logits[(long long)row * V + v] = sum;
                if (row == 1 && dl) dl[v] = sum;
                if (row == 0) {
                    if (sum > bv0 || (sum == bv0 && v < bi0)) { bv0 = sum; bi0 = v; }
                } else {
                    if (sum > bv1 || (sum == bv1 && v < bi1)) { bv1 = sum; bi1 = v; }
                }
            }
        }
        __syncthreads();
    }
    // CTA argmax (threads 0..2RG-1 hold candidates; even threads row 0, odd row 1)
    {
        float bv = (threadIdx.x & 1) ? bv1 : bv0;
        int bi = (threadIdx.x & 1) ? bi1 : bi0;
        if (threadIdx.x >= 2 * RG) { bv = -INFINITY; bi = 0x7fffffff; }
        // reduce within warp 0 separately per parity
        if (warp == 0) {
#pragma unroll
            for (int o = 16; o >= 2; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
            }
            if (lane < 2) {
                P->lm_part[blockIdx.x * 4 + lane * 2] = bv;
                P->lm_part[blockIdx.x * 4 + lane * 2 + 1] = __int_as_float(bi);
            }
        }
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(P->lm_cnt, 1) == (int)gridDim.x - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // last CTA: combine CTA candidates in CTA order (ties to the lower id)
    for (int row = 0; row < 2; ++row) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        for (int c = threadIdx.x; c < (int)gridDim.x; c += blockDim.x) {
            const float v = __ldcg(P->lm_part + c * 4 + row * 2);
            const int i = __float_as_int(__ldcg(P->lm_part + c * 4 + row * 2 + 1));
            if (v > bv || (v == bv && i < bi)) { bv = v; bi = i; }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if (lane == 0) { s_bv[row][warp] = bv; s_bi[row][warp] = bi; }
    }
    __syncthreads();
    if (threadIdx.x < 2) {
        const int row = threadIdx.x;
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        for (int w = 0; w < GEMV_WARPS; ++w) {
            const float v = s_bv[row][w];
            const int i = s_bi[row][w];
            if (v > bv || (v == bv && i < bi)) { bv = v; bi = i; }
        }
        P->st->top[row] = bi;
        P->st->topval[row] = bv;
    }
    if (threadIdx.x == 0) *P->lm_cnt = 0;
}

// ---------------------------------------------------------------------------------
template <typename T>
void launch_target_qkv(const Plan *P, const Plan &h, int round, int grid, cudaStream_t s) {
    k_target_gemv<T, EPI_QKV><<<grid, GEMV_THREADS, h.d * sizeof(float), s>>>(P, round);
}
template <typename T>
void launch_target_oproj(const Plan *P, const Plan &h, int round, int grid, cudaStream_t s) {
    k_target_gemv<T, EPI_OPROJ><<<grid, GEMV_THREADS, h.q_rows * sizeof(float), s>>>(P, round);
}
template <typename T>
void launch_target_gateup(const Plan *P, const Plan &h, int round, int grid, cudaStream_t s) {
    k_target_gemv<T, EPI_GATEUP><<<grid, GEMV_THREADS, h.d * sizeof(float), s>>>(P, round);
}
template <typename T>
void launch_target_down(const Plan *P, const Plan &h, int round, int grid, cudaStream_t s) {
    k_target_gemv<T, EPI_DOWN><<<grid, GEMV_THREADS, h.F * sizeof(float), s>>>(P, round);
}
template <typename T>
void launch_lm_head(const Plan *P, const Plan &h, int grid, cudaStream_t s) {
    if (h.pdm_lm_head == h.lm_head)
        k_lm_head<T, true><<<grid, GEMV_THREADS, 2 * h.d * sizeof(float), s>>>(P);
    else
        k_lm_head<T, false><<<grid, GEMV_THREADS, 2 * h.d * sizeof(float), s>>>(P);
}

int target_blocks_per_sm(int dtype, int smem) {
    int b = 0;
    if (dtype == SPD_BF16)
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_target_gemv<__nv_bfloat16, EPI_DOWN>, GEMV_THREADS, smem);
    else
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_target_gemv<float, EPI_DOWN>, GEMV_THREADS, smem);
    return b > 0 ? b : 1;
}
int lm_blocks_per_sm(int dtype, int smem, bool tied) {
    int b = 0;
    if (dtype == SPD_BF16) {
        if (tied) cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_lm_head<__nv_bfloat16, true>, GEMV_THREADS, smem);
        else cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_lm_head<__nv_bfloat16, false>, GEMV_THREADS, smem);
    } else {
        if (tied) cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_lm_head<float, true>, GEMV_THREADS, smem);
        else cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_lm_head<float, false>, GEMV_THREADS, smem);
    }
    return b > 0 ? b : 1;
}

int gemv_smem_bytes(const Plan &h) {
    int m = h.d;
    if (h.q_rows > m) m = h.q_rows;
    if (h.F > m) m = h.F;
    if (2 * h.d > m) m = 2 * h.d;
    return m * (int)sizeof(float);
}

void set_target_attributes(int smem) {
    cudaFuncSetAttribute(k_target_gemv<float, EPI_QKV>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaFuncSetAttribute(k_target_gemv<float, EPI_OPROJ>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaFuncSetAttribute(k_target_gemv<float, EPI_GATEUP>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaFuncSetAttribute(k_target_gemv<float, EPI_DOWN>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaFuncSetAttribute(k_target_gemv<__nv_bfloat16, EPI_QKV>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaFuncSetAttribute(k_target_gemv<__nv_bfloat16, EPI_OPROJ>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaFuncSetAttribute(k_target_gemv<__nv_bfloat16, EPI_GATEUP>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaFuncSetAttribute(k_target_gemv<__nv_bfloat16, EPI_DOWN>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaFuncSetAttribute(k_lm_head<float, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaFuncSetAttribute(k_lm_head<float, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaFuncSetAttribute(k_lm_head<__nv_bfloat16, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaFuncSetAttribute(k_lm_head<__nv_bfloat16, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

#define INST(T)                                                                                   \
    template void launch_target_qkv<T>(const Plan *, const Plan &, int, int, cudaStream_t);       \
    template void launch_target_oproj<T>(const Plan *, const Plan &, int, int, cudaStream_t);     \
    template void launch_target_gateup<T>(const Plan *, const Plan &, int, int, cudaStream_t);    \
    template void launch_target_down<T>(const Plan *, const Plan &, int, int, cudaStream_t);      \
    template void launch_lm_head<T>(const Plan *, const Plan &, int, cudaStream_t);
INST(float)
INST(__nv_bfloat16)
#undef INST

}  // namespace spd
