// K4 placeholder until the tensor-core prefill kernel lands.
#include "pkv.h"

extern "C" int pkv_paged_prefill_attention(void *, const void *, const int32_t *, int, int, int, const void *,
                                           const void *, const int32_t *, int, const int32_t *, int, int, int, int,
                                           int, float, int, int, int *, void *) {
    return PKV_ERR_UNSUPPORTED;
}
