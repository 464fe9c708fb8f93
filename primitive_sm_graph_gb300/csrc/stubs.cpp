// Entry points whose kernels are not written yet: they refuse every call.
#include "common.h"

extern "C" {

psg_status psg_query_launch(int, const psg_view*, int*, int*, int*, int*)
{
    return PSG_E_UNSUPPORTED_LAYOUT;
}

}  // extern "C"
