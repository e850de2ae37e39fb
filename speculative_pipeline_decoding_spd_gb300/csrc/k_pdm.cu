// Draft-module kernels, the draft GEMM plan, and the tensor-core LM head.
//
// The draft module runs on a second stream, concurrent with the target's rounds: one
// launch per GEMM (one CTA per SM, the CTA code in pdm.cuh) and one per attention
// (k_attn.cu).  Its rows' inputs are the step's input states, so nothing in it waits for
// the target's rounds of the same step; the LM head waits for both streams.  With bf16
// weights and a tied head the LM head is the same GEMM over two rows (OP_LM), each given as
// two bf16 parts (the value and the rest) whose products are added.
#include "pdm.cuh"

namespace spd {

template <typename T, int OP, int MT>
__global__ void __launch_bounds__(PG_THREADS, 1) k_pdm_gemm(const Plan *__restrict__ P, int layer) {
    extern __shared__ __align__(128) unsigned char pg_smem[];
    __shared__ __align__(8) uint64_t full[PG_MAXNS], empty[PG_MAXNS], xbar;
    __shared__ PdmRows pr;
    __shared__ float s_inv[MAXS];
    __shared__ int s_done, s_flag;
    if (threadIdx.x < 32) {
        warp_pdm_rows(P, pr, &s_done);
        if (threadIdx.x == 0) {
            for (int i = 0; i < PG_MAXNS; ++i) {
                mbar_init(&full[i], 1);
                mbar_init(&empty[i], PG_CONSUMERS / 32);
            }
            mbar_init(&xbar, 1);
            fence_mbar_init();
        }
    }
    __syncthreads();
    if (s_done) return;
    pdm_gemm_cta<T, OP, MT>(P, pr, layer, blockIdx.x, gridDim.x, pg_smem, full, empty, &xbar, s_inv, &s_flag);
}

// ---------------------------------------------------------------------------------
// Host side: K slab width per GEMM so that the x rows of one slab fit their budget.
static int pg_slab(int K, int rows, int esz) {
    int kx = pg_round(K, PG_KB);
    int ns = 1;
    while (pg_xbytes(rows, kx, esz) > PG_XMAX) {
        ++ns;
        kx = pg_round((K + ns - 1) / ns, PG_KB);
    }
    return kx;
}

void pdm_plan(int d, int F, int q_rows, int nB, int n, int dtype, int kx[6], int ns[6], int *MT) {
    const int esz = dtype == SPD_BF16 ? 2 : 4, rows = n + 1;
    *MT = rows <= 16 ? 1 : 2;
    const int Ks[6] = {nB * d, d, q_rows, d, F, d};
    for (int i = 0; i < 6; ++i) {
        // bf16: every row as two bf16 parts (the LM head: two rows, each as two parts)
        kx[i] = pg_slab(Ks[i], i == OP_LM ? 4 : (esz == 2 ? 2 * rows : rows), esz);
        ns[i] = (Ks[i] + kx[i] - 1) / kx[i];
    }
}

template <typename T, int OP, int MT>
static void pg_launch(const Plan *P, const Plan &h, int layer, int grid, cudaStream_t s) {
    // the projection opens the draft stream's step (it follows the fork from the target's
    // stream): a full dependency; the rest may start while their predecessor drains
    launch_k(k_pdm_gemm<T, OP, MT>, dim3(grid), dim3(PG_THREADS), PG_SMEM, s, h.pdl != 0 && OP != OP_PROJ, P, layer);
}

template <typename T, int MT>
static void pdm_step_mt(const Plan *P, const Plan &h, int grid, cudaStream_t s) {
    pg_launch<T, OP_PROJ, MT>(P, h, 0, grid, s);
    for (int li = 0; li < h.Ls; ++li) {
        pg_launch<T, OP_QKV, MT>(P, h, li, grid, s);
        launch_pdm_attn<T>(P, h, li, s);
        pg_launch<T, OP_OPROJ, MT>(P, h, li, grid, s);
        pg_launch<T, OP_GATEUP, MT>(P, h, li, grid, s);
        pg_launch<T, OP_DOWN, MT>(P, h, li, grid, s);
    }
}

// The tied bf16 LM head (two rows, one K slab: V % 8 == 0 and x of both rows in shared memory).
bool lm_on_tensor_cores(const Plan &h) {
    return h.dtype == SPD_BF16 && h.pdm_lm_head == h.lm_head && h.V % 8 == 0 && h.pdm_ns[OP_LM] == 1;
}

template <typename T>
void launch_pdm_lm(const Plan *P, const Plan &h, int grid, cudaStream_t s) {
    launch_k(k_pdm_gemm<T, OP_LM, 1>, dim3(grid), dim3(PG_THREADS), PG_SMEM, s, h.pdl != 0, P, 0);
}

template <typename T>
void launch_pdm_step(const Plan *P, const Plan &h, int grid, cudaStream_t s) {
    if (h.pdm_MT == 1) pdm_step_mt<T, 1>(P, h, grid, s);
    else pdm_step_mt<T, 2>(P, h, grid, s);
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
    cudaFuncSetAttribute(k_pdm_gemm<float, OP_LM, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, PG_SMEM);
    cudaFuncSetAttribute(k_pdm_gemm<__nv_bfloat16, OP_LM, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, PG_SMEM);
    set_attr_mt<float, 1>();
    set_attr_mt<float, 2>();
    set_attr_mt<__nv_bfloat16, 1>();
    set_attr_mt<__nv_bfloat16, 2>();
}

template void launch_pdm_step<float>(const Plan *, const Plan &, int, cudaStream_t);
template void launch_pdm_lm<float>(const Plan *, const Plan &, int, cudaStream_t);
template void launch_pdm_lm<__nv_bfloat16>(const Plan *, const Plan &, int, cudaStream_t);
template void launch_pdm_step<__nv_bfloat16>(const Plan *, const Plan &, int, cudaStream_t);

}  // namespace spd
