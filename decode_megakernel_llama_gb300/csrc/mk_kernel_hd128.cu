// mk_kernel_hd128.cu — megakernel instances for head dimension 128
// (G = 1..4 query heads per kv head), compiled as their own translation unit.
#include "mk_kernel.cuh"

extern "C" const void *mk_kernel_fn_hd128(int G) {
    switch (G) {
        case 1: return (const void *)mk::mk_megakernel<128, 1, false>;
        case 2: return (const void *)mk::mk_megakernel<128, 2, false>;
        case 3: return (const void *)mk::mk_megakernel<128, 3, false>;
        case 4: return (const void *)mk::mk_megakernel<128, 4, false>;
        default: return nullptr;
    }
}
