// gemv_f32.cu -- fp32-weight instantiations of the fused GEMV (gemv_impl.cuh).
#include "gemv_impl.cuh"

namespace gd {

const void* gemv_kernel_f32(int nr, int cpl, int pro, int epi) {
    if (nr == 1) {
        switch (cpl) {
            case 0: return gemv_pick_epi<float, 1, 0>(pro, epi);
            case 1: return gemv_pick_epi<float, 1, 1>(pro, epi);
            case 2: return gemv_pick_epi<float, 1, 2>(pro, epi);
        }
    } else if (nr == 4) {
        if (cpl == 0) return gemv_pick_epi<float, 4, 0>(pro, epi);
        if (cpl == 1) return gemv_pick_epi<float, 4, 1>(pro, epi);
    } else if (nr == 8) {
        if (cpl == 0) return gemv_pick_epi<float, 8, 0>(pro, epi);
    }
    return nullptr;
}

}  // namespace gd
