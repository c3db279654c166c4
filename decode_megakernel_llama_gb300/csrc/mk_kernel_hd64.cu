// mk_kernel_hd64.cu — megakernel instances for head dimension 64
// (G = 1..4 query heads per kv head), compiled as their own translation unit.
#include "mk_kernel.cuh"

extern "C" const void *mk_kernel_fn_hd64(int G) {
    switch (G) {
        case 1: return (const void *)mk::mk_megakernel<64, 1, false>;
        case 2: return (const void *)mk::mk_megakernel<64, 2, false>;
        case 3: return (const void *)mk::mk_megakernel<64, 3, false>;
        case 4: return (const void *)mk::mk_megakernel<64, 4, false>;
        default: return nullptr;
    }
}

// Batched-step instances (hd 64 only).
extern "C" const void *mk_kernel_fn_hd64_batch(int G) {
    switch (G) {
        case 1: return (const void *)mk::mk_megakernel<64, 1, true>;
        case 2: return (const void *)mk::mk_megakernel<64, 2, true>;
        case 3: return (const void *)mk::mk_megakernel<64, 3, true>;
        case 4: return (const void *)mk::mk_megakernel<64, 4, true>;
        default: return nullptr;
    }
}
