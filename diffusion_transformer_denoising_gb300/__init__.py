"""GB300-native denoiser stage: DiT forward loop + classifier-free guidance +
flow-matching Euler, behind a C ABI (libdit.so) with hand-written sm_103a
kernels.  The binding in `dit` loads the library on first use and fails
loudly if it has not been built."""
