// Host-side helpers shared by the C-ABI translation units.
#pragma once

namespace pkv {
// Records a printf-style message for pkv_last_error() on this thread and returns code.
int set_error(int code, const char* fmt, ...);
}  // namespace pkv
