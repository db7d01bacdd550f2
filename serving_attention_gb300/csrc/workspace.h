// workspace.h -- int workspace geometry shared by the planner and the run
// entry points (C++ only; the layout itself is in plan_layout.h).
#pragma once
#include <stdint.h>

#include "../../include/fi.h"

namespace fi {

// int32 slots of the plan region at the config's capacities (header, CTA
// offsets, items, merge units, counters, requests); the RoPE table follows
// at fi_rope_table_offset() of this.
int64_t plan_capacity_ints(const fi_plan_config* cfg);

}  // namespace fi
