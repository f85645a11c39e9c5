// Host-side helpers shared by the library's translation units.
#pragma once

namespace specv {

// SPEC_OK when the current device is an sm_103 GPU, SPEC_E_ARCH otherwise,
// SPEC_E_CUDA when the device cannot be queried.  Cached per device.
int check_arch();

}  // namespace specv
