// Frequency-admitted HBM expert cache: placeholder until the step-end pass lands.
#include "internal.h"

cudaError_t moe::lfu_step_end(Plan&, cudaStream_t) { return cudaErrorNotSupported; }
