// gemv.cu -- host-side planning and launch of the fused GEMV kernels
// (gemv_impl.cuh; instantiated in gemv_bf16.cu and gemv_f32.cu).
#include "common.cuh"
#include "internal.h"

namespace gd {

const void* gemv_kernel_bf16(int nr, int cpl, int pro, int epi);
const void* gemv_kernel_f32(int nr, int cpl, int pro, int epi);
const void* gemv_tc_kernel(int pro, int epi, int ws);
cudaError_t gemv_tc_plan(GemvPlan* plan, int num_sms);
const void* gemv_box_kernel(int pro, int epi);
cudaError_t gemv_box_plan(GemvPlan* plan, int num_sms);
cudaError_t gemv_box_launch(const GemvPlan& plan, cudaStream_t s, bool pdl);

namespace {
// mirrors gemv_impl.cuh
constexpr int SL = 8;                    // K-slices
constexpr int GR = 1;                    // row groups
constexpr int THREADS = SL * GR * 32;
constexpr int STAGE_MAX = 32768;         // bytes per ring stage at most
constexpr int MAX_S = 6;
constexpr int MAX_RPS = 32;

const void* pick(const GemvPlan& pl) {
    if (pl.tc == 2) return gemv_box_kernel(pl.pro, pl.epi);
    if (pl.tc) return gemv_tc_kernel(pl.pro, pl.epi, pl.p.tc_ws);
    return pl.wtype == W_BF16 ? gemv_kernel_bf16(pl.nr, pl.cpl, pl.pro, pl.epi)
                              : gemv_kernel_f32(pl.nr, pl.cpl, pl.pro, pl.epi);
}

// register-resident activation chunks per lane: the instantiated value >= need
int cpl_for(int need, int nr, int wtype) {
    const int opts_bf16_1[] = {1, 2, 4, 7};
    if (need <= 0) return 0;
    if (wtype == W_BF16 && nr == 1) {
        for (int o : opts_bf16_1)
            if (o >= need) return o;
        return 0;
    }
    if (wtype == W_BF16 && nr == 4) return need <= 1 ? 1 : (need <= 2 ? 2 : 0);
    if (wtype == W_BF16 && nr == 8) return need <= 1 ? 1 : 0;
    if (wtype == W_F32 && nr == 1) return need <= 1 ? 1 : (need <= 2 ? 2 : 0);
    if (wtype == W_F32 && nr == 4) return need <= 1 ? 1 : 0;
    return 0;
}
}  // namespace

cudaError_t gemv_plan(GemvPlan* plan, int num_sms) {
    if (plan->tc == 2) {
        // box-streamed tensor-core GEMV; the row-copy one where no box plan fits
        if (gemv_box_plan(plan, num_sms) == cudaSuccess) return cudaSuccess;
        plan->tc = 1;
    }
    if (plan->tc) return gemv_tc_plan(plan, num_sms);
    GemvParams& p = plan->p;
    const int vec = plan->wtype == W_BF16 ? 8 : 4;
    const int es = plan->wtype == W_BF16 ? 2 : 4;
    if (p.K <= 0 || p.N <= 0 || p.R < 1 || p.R > 8) return cudaErrorInvalidValue;
    if (p.K % (SL * vec) != 0) return cudaErrorInvalidValue;              // whole vectors per K-slice
    if ((size_t)p.K * es > (size_t)STAGE_MAX) return cudaErrorInvalidValue;  // a row fits one stage
    plan->nr = p.R == 1 ? 1 : (p.R <= 4 ? 4 : 8);
    const int swv = p.K / (SL * vec);
    const int need = (swv + 31) / 32;
    plan->cpl = cpl_for(need, plan->nr, plan->wtype);
    const void* fn = pick(*plan);
    if (!fn) return cudaErrorInvalidValue;
    // rows per stage: a whole number of rows in <= 64 KB (<= 32 KB when the
    // activations also live in shared memory), a multiple of the rows the two
    // row groups load together (2 * 8 / cpl)
    const size_t stage_cap = (size_t)STAGE_MAX;
    int rps = (int)(stage_cap / ((size_t)p.K * es));
    if (rps > MAX_RPS) rps = MAX_RPS;
    const int ru = plan->cpl == 0 ? 2 : (8 / plan->cpl > 0 ? 8 / plan->cpl : 1);
    if (rps >= GR * ru) rps -= rps % (GR * ru);
    else if (rps >= GR) rps -= rps % GR;
    p.rps = rps < 1 ? 1 : rps;
    const size_t stage_bytes = (size_t)p.rps * p.K * es;
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) return e;
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, fn)) != cudaSuccess) return e;
    const size_t avail = (size_t)optin - fa.sharedSizeBytes;
    const size_t act = plan->cpl == 0 ? (size_t)plan->nr * p.K * sizeof(float) : 0;
    // ring depth: ~96 KB, so that two CTAs (this kernel's and the next one's,
    // launched early by the programmatic edge) fit on an SM together
    int S = (int)(98304 / stage_bytes);
    if (S > MAX_S) S = MAX_S;
    if (S < 2) S = 2;
    while (S > 2 && (size_t)S * stage_bytes + act > avail) --S;
    if (plan->cpl == 0) plan->grid = p.N < num_sms ? p.N : num_sms;   // activations in smem: one CTA per SM
    if ((size_t)S * stage_bytes + act > avail) return cudaErrorInvalidValue;
    p.stages = S;
    plan->smem = (size_t)S * stage_bytes + act;
    plan->block = THREADS;
    plan->grid = p.N < 2 * num_sms ? p.N : 2 * num_sms;
    return raise_smem_cap(fn);
}

cudaError_t gemv_launch(const GemvPlan& plan, cudaStream_t s, bool pdl) {
    if (plan.tc == 2) return gemv_box_launch(plan, s, pdl);
    const void* fn = pick(plan);
    if (!fn) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.grid);
    cfg.blockDim = dim3(plan.block);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    void* args[] = {const_cast<GemvParams*>(&plan.p)};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace gd
