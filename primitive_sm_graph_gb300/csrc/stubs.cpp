// Entry points whose kernels are not written yet: they refuse every call.
#include "common.h"

extern "C" {

psg_status psg_contract(const void*, const psg_view*, const void*, const psg_view*, void*,
                        const psg_view*, int32_t*, void*)
{
    return PSG_E_UNSUPPORTED_LAYOUT;
}
psg_status psg_query_launch(int, const psg_view*, int*, int*, int*, int*)
{
    return PSG_E_UNSUPPORTED_LAYOUT;
}

}  // extern "C"
