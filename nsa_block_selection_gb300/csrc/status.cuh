// Per-translation-unit device status words (bounded waits that gave up),
// read and cleared by nsa_sync_status. Internal; not part of the public ABI.
#pragma once

namespace nsa {

int fwd_read_and_clear_status(unsigned int* value);  // selection forward (+ wait self-test)
int bwd_read_and_clear_status(unsigned int* value);  // selection backward
int swa_read_and_clear_status(unsigned int* value);  // sliding-window forward
int shared_read_and_clear_status(unsigned int* value);  // tile-shared pass of the forward
int probe_read_and_clear_status(unsigned int* value);   // gather-bandwidth probe

}  // namespace nsa
