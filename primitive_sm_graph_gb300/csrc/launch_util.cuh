// Launch helpers: SM count, occupancy and register counts, cached per device.
#pragma once

#include <algorithm>
#include <cstdint>

namespace psg {

int current_device();
int num_sms();                                                 // of the current device
int max_blocks_per_sm(const void* fn, int threads, size_t smem);  // occupancy, >= 1
int kernel_regs(const void* fn);
size_t l2_bytes();

}  // namespace psg
