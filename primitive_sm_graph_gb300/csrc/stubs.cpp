// Entry points whose kernels are not written yet: they refuse every call.
#include "common.h"

extern "C" {

psg_status psg_contract(const void*, const psg_view*, const void*, const psg_view*, void*,
                        const psg_view*, int32_t*, void*)
{
    return PSG_E_UNSUPPORTED_LAYOUT;
}
psg_status psg_gather(const void*, const psg_view*, const int32_t*, int64_t, void*,
                      const psg_view*, int32_t*, void*)
{
    return PSG_E_UNSUPPORTED_LAYOUT;
}
size_t psg_scatter_workspace(int64_t) { return 0; }
psg_status psg_scatter_add(void*, const psg_view*, const int32_t*, int64_t, const void*,
                           const psg_view*, void*, size_t, int32_t*, void*)
{
    return PSG_E_UNSUPPORTED_LAYOUT;
}
psg_status psg_query_launch(int, const psg_view*, int*, int*, int*, int*)
{
    return PSG_E_UNSUPPORTED_LAYOUT;
}

}  // extern "C"
