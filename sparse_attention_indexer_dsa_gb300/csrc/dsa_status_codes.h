// Codes the device writes into the workspace status word.  They equal the
// public dsa_status_t values of include/dsa_idx.h.
#pragma once
#define DSA_DEV_OK 0
#define DSA_DEV_ERR_INVALID_ARG 1
#define DSA_DEV_ERR_TIMEOUT 5
#define DSA_DEV_ERR_BOUNDS 6   // checked build only: a device-side bounds check failed
