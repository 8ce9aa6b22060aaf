// decode_f16.cu -- fp16 instantiations of the decode kernel.
#include "decode.cuh"

namespace pkv {

DecodeKernelInfo decode_info_f16(int head_dim, int gs) {
    using T = __half;
    DecodeKernelInfo none{nullptr, 0, 0, 0, 0};
    if (head_dim == 128) {
        switch (gs) {
            case 1: return make_decode_info<T, 128, 1>();
            case 2: return make_decode_info<T, 128, 2>();
            case 3: return make_decode_info<T, 128, 3>();
            case 4: return make_decode_info<T, 128, 4>();
            case 5: return make_decode_info<T, 128, 5>();
            case 6: return make_decode_info<T, 128, 6>();
            case 7: return make_decode_info<T, 128, 7>();
            case 8: return make_decode_info<T, 128, 8>();
        }
    } else if (head_dim == 64) {
        switch (gs) {
            case 1: return make_decode_info<T, 64, 1>();
            case 2: return make_decode_info<T, 64, 2>();
            case 3: return make_decode_info<T, 64, 3>();
            case 4: return make_decode_info<T, 64, 4>();
            case 5: return make_decode_info<T, 64, 5>();
            case 6: return make_decode_info<T, 64, 6>();
            case 7: return make_decode_info<T, 64, 7>();
            case 8: return make_decode_info<T, 64, 8>();
        }
    }
    return none;
}

}  // namespace pkv
