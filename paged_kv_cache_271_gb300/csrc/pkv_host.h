// Host-side helpers shared by the C-ABI translation units.
#pragma once

namespace pkv {
// Records a printf-style message for pkv_last_error() on this thread and returns code.
int set_error(int code, const char* fmt, ...);
// The driver's current context on this host thread, as an opaque handle (nullptr: none is
// current, or the driver's entry point could not be found).
void* current_context();
// Makes the current device's primary context current on this host thread when no context is.
// The runtime binds it to a thread only at the first runtime call that needs it, and a driver
// call made before that (the tensor-map encoder) fails with an invalid-context error. A context
// that is already current is left as it is. Returns PKV_OK or a PKV_ECUDA status.
int bind_context(const char* who);
}  // namespace pkv
