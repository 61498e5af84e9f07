// The opaque muon_layout handle of the C ABI: the host plan and, once a GPU call has
// prepared it, the device tables.
#pragma once

#include <mutex>

#include "kernels.h"
#include "muon_internal.h"

struct muon_layout {
  muon::Plan plan;
  muon::DevTables dt;
  std::mutex mu;
};
