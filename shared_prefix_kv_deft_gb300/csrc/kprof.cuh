// kprof.cuh -- optional in-kernel timestamps for development builds.
//
// Compiled out unless DEFT_KPROF is defined.  When defined, KPROF(args, slot)
// stores %globaltimer (ns) into args.kprof[slot] from the first CTA of a
// launch only; capi.cu owns the buffer and deft_kprof_read() copies it out.
#pragma once

#include <stdint.h>

namespace deft {
constexpr int kKprofSlots = 4096;
// The timestamp buffer alone, for kernels that take no AttnArgs.
struct KprofArg {
    unsigned long long *kprof;
};
}

#ifdef DEFT_KPROF
#define KPROF(args, slot)                                                            \
    do {                                                                             \
        if (blockIdx.x == 0 && (args).kprof && (slot) >= 0 &&                       \
            (slot) < ::deft::kKprofSlots) {                                          \
            unsigned long long t_;                                                   \
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));                    \
            (args).kprof[(slot)] = t_;                                               \
        }                                                                            \
    } while (0)
// KPROF_ANY: the same from any CTA.
#define KPROF_ANY(args, slot)                                                        \
    do {                                                                             \
        if ((args).kprof && (slot) >= 0 && (slot) < ::deft::kKprofSlots) {          \
            unsigned long long t_;                                                   \
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));                    \
            (args).kprof[(slot)] = t_;                                               \
        }                                                                            \
    } while (0)
#else
#define KPROF_ANY(args, slot) \
    do {                      \
    } while (0)
#define KPROF(args, slot) \
    do {                  \
    } while (0)
#endif
