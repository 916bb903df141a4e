// Shared host-side helpers of the library (error reporting).
#pragma once
#include <string>

namespace qmoe {
// Records `msg` as the calling thread's last error and returns `status`.
int fail(int status, const std::string& msg);
void clear_error();
const char* last_error();
}  // namespace qmoe
