// Internal helpers shared by the host-side sources of the library.
#pragma once

#include <cstdint>

#include "mb.h"

namespace mb {

// Record a message for mb_last_error() and return `st`.
mb_status fail(mb_status st, const char *fmt, ...);

}  // namespace mb
