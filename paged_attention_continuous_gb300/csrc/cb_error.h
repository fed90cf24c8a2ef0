// Thread-local error message shared by every translation unit of the C ABI.
#pragma once

#include <cstdarg>
#include <cstdio>
#include <string>

#include "../../include/cb.h"

namespace cb {

std::string& last_error_slot();

inline cb_status fail(cb_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  last_error_slot() = buf;
  return st;
}

inline cb_status ok() { return CB_OK; }

}  // namespace cb
