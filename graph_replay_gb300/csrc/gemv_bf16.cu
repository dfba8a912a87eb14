// gemv_bf16.cu -- bf16-weight instantiations of the fused GEMV (gemv_impl.cuh).
#include "gemv_impl.cuh"

namespace gd {

const void* gemv_kernel_bf16(int nr, int cpl, int pro, int epi) {
    using T = __nv_bfloat16;
    if (nr == 1) {
        switch (cpl) {
            case 0: return gemv_pick_epi<T, 1, 0>(pro, epi);
            case 1: return gemv_pick_epi<T, 1, 1>(pro, epi);
            case 2: return gemv_pick_epi<T, 1, 2>(pro, epi);
            case 4: return gemv_pick_epi<T, 1, 4>(pro, epi);
            case 7: return gemv_pick_epi<T, 1, 7>(pro, epi);
        }
    } else if (nr == 4) {
        switch (cpl) {
            case 0: return gemv_pick_epi<T, 4, 0>(pro, epi);
            case 1: return gemv_pick_epi<T, 4, 1>(pro, epi);
            case 2: return gemv_pick_epi<T, 4, 2>(pro, epi);
        }
    } else if (nr == 8) {
        switch (cpl) {
            case 0: return gemv_pick_epi<T, 8, 0>(pro, epi);
            case 1: return gemv_pick_epi<T, 8, 1>(pro, epi);
        }
    }
    return nullptr;
}

}  // namespace gd
