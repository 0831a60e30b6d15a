// Prefill-batch forward (T > 8): placeholder until the grouped GEMM lands.
#include "internal.h"
