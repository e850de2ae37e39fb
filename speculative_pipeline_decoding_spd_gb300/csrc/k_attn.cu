// Decode attention of one pipeline step.
//
// Target mode: each occupied stage's token attends, in the layer its stage runs at this
// round, to KV positions 0..pos (machine review "The reading": the n tokens of one
// sequence advance in parallel; the staircase guarantees that every earlier position
// already holds this layer's K,V).  RoPE of q and k and the KV append at pos are fused
// here; the QKV GEMV leaves raw projections.
// Draft mode: the draft module's rows (consecutive positions) attend causally to its
// own KV cache, whose entries for the rows were written by the QKV epilogue.
//
// The attention arithmetic itself (split-K over 128-position chunks, deterministic
// merge) lives in attn.cuh.
#include "attn.cuh"

namespace spd {

// Plan-driven launch: problems are the occupied stages with a layer at this round
// (TARGET, round `arg`) or the draft module's rows at draft layer `arg` (their K,V were
// appended by the draft QKV epilogue).
template <typename T, bool TARGET>
__global__ void __launch_bounds__(ATT_THREADS, att_min_blocks<KvT<T>>()) k_attn(const Plan *__restrict__ P, int arg) {
    using KV = KvT<T>;
    __shared__ int s_ok, s_pos, s_layer, s_src;
    const int Hkv = P->Hkv, hd = P->hd;
    const int g = blockIdx.x % Hkv, c = blockIdx.x / Hkv, prob = blockIdx.y;
    if (threadIdx.x < 32) {
        __shared__ StageList SL;
        __shared__ PdmRows PR;
        __shared__ int s_dn;
        int ok, pos = 0, layer = 0, src = 0;
        if (TARGET) {
            warp_stage_list(P, arg, SL, &s_dn);
            ok = !s_dn && prob < SL.m;
            if (ok) {
                pos = SL.pos[prob];
                layer = SL.layer[prob];
                src = SL.stage[prob];
            }
        } else {
            warp_pdm_rows(P, PR, &s_dn);
            ok = !s_dn && prob < PR.R;
            pos = PR.pos0 + prob;
            layer = arg;
            src = prob;
        }
        if (ok && c * ATT_CHUNK > pos) ok = 0;
        if (threadIdx.x == 0) {
            s_ok = ok;
            s_pos = pos;
            s_layer = layer;
            s_src = src;
        }
    }
    __syncthreads();
    if (!s_ok) return;
    if (!TARGET) pdl_wait();   // the rows' K,V were appended by the preceding draft QKV launch
    AttnArgs<KV> a{};
    const long long kvoff = (long long)s_layer * P->kv_stride;
    a.kc = reinterpret_cast<KV *>(TARGET ? P->kc : P->pkc) + kvoff;
    a.vc = reinterpret_cast<KV *>(TARGET ? P->vc : P->pvc) + kvoff;
    a.S = s_pos + 1;
    a.maxch = P->att_max_chunks;
    a.Hq = P->Hq;
    a.Hkv = Hkv;
    a.hd = hd;
    a.scale = P->scale;
    if (TARGET) {
        const float *raw = P->QKV + (long long)s_src * P->qkv_rows;
        a.q = raw;
        a.rope = P->rope + (long long)s_pos * (hd / 2);
        a.kraw = raw + P->q_rows;
        a.vraw = raw + P->q_rows + P->kv_rows;
        a.out = nullptr;
        a.part = P->att_part;
        a.cnt = nullptr;   // the O projection merges the chunks while staging its input
        a.prob = s_src;    // partials indexed by stage
    } else {
        a.q = P->QKVp + (long long)s_src * P->qkv_rows;
        a.rope = nullptr;
        a.kraw = nullptr;
        a.vraw = nullptr;
        // bf16 weights: the O GEMM copies its input rows as two bf16 parts
        if (sizeof(T) == 2) {
            a.outb = P->ATTb + (long long)s_src * P->q_rows;
            a.outb_lo = (long long)(P->n + 1) * P->q_rows;
        } else {
            a.out = P->ATTp + (long long)s_src * P->q_rows;
        }
        a.part = P->patt_part;
        a.cnt = P->patt_cnt;
        a.prob = s_src;
    }
    attn_cta<KV>(a, g, c);
}

int attn_smem_bytes(int dtype, int hd, int G) {
    return dtype == SPD_BF16 ? att_smem_bytes<KvT<__nv_bfloat16>>(hd, G) : att_smem_bytes<float>(hd, G);
}

void set_attn_attributes() {
    cudaFuncSetAttribute(k_attn<float, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         att_smem_bytes<float>(ATT_MAXHD, ATT_MAXG));
    cudaFuncSetAttribute(k_attn<float, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         att_smem_bytes<float>(ATT_MAXHD, ATT_MAXG));
    cudaFuncSetAttribute(k_attn<__nv_bfloat16, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         att_smem_bytes<KvT<__nv_bfloat16>>(ATT_MAXHD, ATT_MAXG));
    cudaFuncSetAttribute(k_attn<__nv_bfloat16, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         att_smem_bytes<KvT<__nv_bfloat16>>(ATT_MAXHD, ATT_MAXG));
    cudaFuncSetAttribute(k_attn<float, true>, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    cudaFuncSetAttribute(k_attn<float, false>, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    cudaFuncSetAttribute(k_attn<__nv_bfloat16, true>, cudaFuncAttributePreferredSharedMemoryCarveout,
                         cudaSharedmemCarveoutMaxShared);
    cudaFuncSetAttribute(k_attn<__nv_bfloat16, false>, cudaFuncAttributePreferredSharedMemoryCarveout,
                         cudaSharedmemCarveoutMaxShared);
}

template <typename T>
void launch_target_attn(const Plan *P, const Plan &h, int round, cudaStream_t s) {
    dim3 grid(h.att_max_chunks * h.Hkv, h.n);
    launch_k(k_attn<T, true>, grid, dim3(ATT_THREADS), att_smem_bytes<KvT<T>>(h.hd, h.Hq / h.Hkv), s, h.pdl != 0, P, round);
}
template <typename T>
void launch_pdm_attn(const Plan *P, const Plan &h, int layer, cudaStream_t s) {
    dim3 grid(h.att_max_chunks * h.Hkv, h.n + 1);
    launch_k(k_attn<T, false>, grid, dim3(ATT_THREADS), att_smem_bytes<KvT<T>>(h.hd, h.Hq / h.Hkv), s, h.pdl != 0, P, layer);
}

template void launch_target_attn<float>(const Plan *, const Plan &, int, cudaStream_t);
template void launch_target_attn<__nv_bfloat16>(const Plan *, const Plan &, int, cudaStream_t);
template void launch_pdm_attn<float>(const Plan *, const Plan &, int, cudaStream_t);
template void launch_pdm_attn<__nv_bfloat16>(const Plan *, const Plan &, int, cudaStream_t);

}  // namespace spd
