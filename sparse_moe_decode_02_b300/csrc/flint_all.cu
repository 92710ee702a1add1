// flint_all.cu -- single translation unit of the Flint library (the device status
// word and the kernels share one module without relocatable device code).
#include "quantize.cu"
#include "decode.cu"
#include "lm_head.cu"
#include "prefill.cu"
#include "mma_bench.cu"
#include "sample.cu"
#include "api.cu"
#include "noalloc.cu"
