// Process-wide debug switches of the library (set through dg_set_debug), shared by every
// translation unit that launches a GEMM kernel.
#pragma once

namespace dg {

// kFault* value every later launch passes to its kernel (0: none).
int debug_fault_mode();

// Limit of every pipeline wait of later launches, in ns (the default unless dg_set_debug set one).
unsigned long long pipeline_wait_timeout_ns();

}  // namespace dg
