// route.h -- host-side choice between the two tile kernels for M above the few-token
// range, and the registry of packed q6_K weights' fold state that the choice reads.
// Host code only; nothing here touches the GPU.
#pragma once

namespace mmq {

// Records that the packed weight at `packed` on device `dev` has this type and shape
// and, for q6_K, whether its codes are folded (fold = 1: one f16 tile sc*q) or split
// in two tiles (fold = 0); fold = -1 forgets any record for that address.  A later
// record for the same address replaces the earlier one.
void note_packed(int dev, const void* packed, int type, int od, int id, int fold);

// The recorded fold state of the packed weight at `packed` (1, 0), or -1 when no
// record matches the address, type and shape.
int packed_fold_state(int dev, const void* packed, int type, int od, int id);

// Whether the super-block kernel should compute Y (else the chunk kernel) for M
// tokens on a device with nsm SMs.  fold is the weight's fold state (q6_K; -1 when
// unknown, taken as folded; q4_K passes 1).
bool prefer_superblock(int type, int od, int id, int M, int nsm, int fold);

}  // namespace mmq
