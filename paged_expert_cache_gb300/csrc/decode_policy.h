// decode_policy.h -- the host's choices of a decode call's path, free of CUDA
// so that they compile and run on their own (the CPU tests do).
//
// Two choices:
//   * which path a decode call takes: one persistent kernel for the whole
//     layer call, or three kernels (route + plan, gate/up, down);
//   * in which form the persistent kernel is launched. Its CTAs wait on one
//     another (grid barriers, the logit announcement), so every CTA must be
//     resident at once: it goes out as a cooperative launch, which the runtime
//     starts only when the whole grid fits. The form with programmatic
//     dependent launch is tried first, then the cooperative launch alone; once
//     both are refused the caller keeps to the three-kernel path.
#pragma once

#include "../../include/moe_cache.h"

namespace moe {

struct DecodeCall {
    int mode;        // moe_decode_mode_t of the handle
    int T;           // tokens of the call
    int pool_mode;   // moe_pool_mode_t
    int upload_mode; // moe_upload_mode_t
    bool speculate;  // the handle prefetches the next layer's experts
    bool fused_ok;   // no launch of the persistent kernel was refused yet
    bool fits;       // the call's shared-memory layout fits one CTA per SM
};

// MOE_DECODE_AUTO takes the one-kernel path for calls of one token, and of
// two tokens on per-layer pools: measured on one GPU it is 3-14% faster there,
// and slower with four tokens or with two tokens on the shared pool, where each
// CTA's redundant ranking and plan, and one CTA per SM streaming more units,
// cost more than the kernel boundaries save. Speculation's side-stream kernels
// run beside the expert kernels, so it keeps to three kernels (the persistent
// kernel holds every SM); so does the MEMCPY upload, whose host copies sit
// between the plan and the expert kernels.
inline bool one_kernel_decode(const DecodeCall& q) {
    if (q.mode == MOE_DECODE_THREE_KERNELS || !q.fused_ok || q.speculate || q.upload_mode != MOE_UPLOAD_PULL ||
        !q.fits)
        return false;
    return q.mode == MOE_DECODE_ONE_KERNEL || q.T == 1 || (q.T == 2 && q.pool_mode == MOE_POOL_PER_LAYER);
}

// Launch forms of the persistent kernel, in the order they are tried.
enum : int { kCoopWithPdl = 0, kCoopAlone = 1, kCoopRefused = 2 };

// Launches through try_form(with_pdl) -> bool, starting from `form` (one
// state per kernel instantiation, kept by the caller). Returns whether a form
// was accepted; a refused form is not tried again. With pdl false the first
// form is the cooperative launch alone, and its refusal is final.
template <class TryForm>
inline bool launch_cooperative(int& form, bool pdl, TryForm&& try_form) {
    if (form == kCoopWithPdl) {
        if (try_form(pdl)) return true;
        form = pdl ? kCoopAlone : kCoopRefused;
    }
    if (form == kCoopAlone) {
        if (try_form(false)) return true;
        form = kCoopRefused;
    }
    return false;
}

}  // namespace moe
