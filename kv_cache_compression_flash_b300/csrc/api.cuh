// Host-side wrapper of every compute entry point of the C ABI:
//  - an NVTX range named after the call (header-only NVTX 3: it costs a
//    branch unless a profiler is attached), so a timeline shows which ABI
//    call enqueued which kernels;
//  - host-side fault injection for tests of the caller's error handling:
//        KVS_FAULT_INJECT=<call>:<code>[,<call>:<code>...]
//    makes the named entry point (e.g. kvs_allocate_bits) return <code>
//    (1..6, see kvs.h) before it validates or enqueues anything.  The
//    variable is read once, at the first call of any entry point.
#pragma once

#include <nvtx3/nvToolsExt.h>

#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include "kvs.h"

namespace kvs {

class ApiScope {
 public:
  explicit ApiScope(const char* name) { nvtxRangePushA(name); }
  ~ApiScope() { nvtxRangePop(); }
  ApiScope(const ApiScope&) = delete;
  ApiScope& operator=(const ApiScope&) = delete;
};

// (call, code) pairs parsed from KVS_FAULT_INJECT; malformed entries are ignored
inline std::vector<std::pair<std::string, int>> parse_fault_inject(const char* spec) {
  std::vector<std::pair<std::string, int>> out;
  if (!spec) return out;
  std::string s(spec);
  size_t pos = 0;
  while (pos <= s.size()) {
    size_t end = s.find(',', pos);
    if (end == std::string::npos) end = s.size();
    const std::string item = s.substr(pos, end - pos);
    const size_t colon = item.rfind(':');
    if (colon != std::string::npos && colon > 0) {
      char* stop = nullptr;
      const long code = std::strtol(item.c_str() + colon + 1, &stop, 10);
      if (stop && *stop == '\0' && code >= KVS_ERR_INVALID_ARG && code <= KVS_ERR_WORKSPACE)
        out.emplace_back(item.substr(0, colon), static_cast<int>(code));
    }
    pos = end + 1;
  }
  return out;
}

inline int injected_fault(const char* call) {
  static std::vector<std::pair<std::string, int>> table;
  static std::once_flag once;
  std::call_once(once, [] { table = parse_fault_inject(std::getenv("KVS_FAULT_INJECT")); });
  for (const auto& e : table)
    if (e.first == call) return e.second;
  return KVS_OK;
}

}  // namespace kvs

// First statement of a compute entry point: its NVTX range, then an injected fault if one is configured.
#define KVS_API_ENTRY()                                \
  const ::kvs::ApiScope kvs_api_scope_(__func__);      \
  if (const int kvs_injected_ = ::kvs::injected_fault(__func__)) return kvs_injected_
