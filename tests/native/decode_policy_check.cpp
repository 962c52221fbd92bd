// Drives the host-side decode policy (decode_policy.h) from stdin, one case
// per line, so the CPU tests can check it without a GPU:
//   path MODE T POOL UPLOAD SPECULATE FUSED_OK FITS   -> prints 1 (one kernel) or 0
//   coop FORM PDL ANSWERS                              -> the runtime's answers to
//        successive launch attempts (A accept, R refuse); prints, per call until
//        the answers run out or a call fails, the forms tried ('p' with PDL, 'c'
//        without), then the result and the form kept for the next call
#include <cstdio>
#include <cstring>
#include <string>
#include "decode_policy.h"

int main() {
    char kind[16];
    while (scanf("%15s", kind) == 1) {
        if (!strcmp(kind, "path")) {
            moe::DecodeCall q;
            int spec, ok, fits;
            if (scanf("%d %d %d %d %d %d %d", &q.mode, &q.T, &q.pool_mode, &q.upload_mode, &spec, &ok, &fits) != 7)
                return 2;
            q.speculate = spec != 0;
            q.fused_ok = ok != 0;
            q.fits = fits != 0;
            printf("%d\n", moe::one_kernel_decode(q) ? 1 : 0);
        } else if (!strcmp(kind, "coop")) {
            int form, pdl;
            char answers[64];
            if (scanf("%d %d %63s", &form, &pdl, answers) != 3) return 2;
            size_t next = 0;
            std::string log;
            bool out_of_answers = false;
            for (;;) {
                std::string tried;
                const bool ok = moe::launch_cooperative(form, pdl != 0, [&](bool with_pdl) {
                    tried += with_pdl ? 'p' : 'c';
                    if (next >= strlen(answers)) {
                        out_of_answers = true;
                        return false;
                    }
                    return answers[next++] == 'A';
                });
                if (out_of_answers) break;
                log += tried + (ok ? ":1:" : ":0:") + std::to_string(form) + " ";
                if (!ok) break;
            }
            printf("%s\n", log.c_str());
        } else {
            return 2;
        }
        fflush(stdout);
    }
    return 0;
}
