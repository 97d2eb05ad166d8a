// Host-side declarations shared between the translation units of libpagedkv.
#pragma once

namespace pkv {

// Number of SMs of the current device (cached per device), or 1 on error.
int num_sms_current();

// Read and clear the sticky device error word of one translation unit.
int append_read_error(unsigned* flags, long long* detail);
int decode_read_error(unsigned* flags, long long* detail);

}  // namespace pkv
