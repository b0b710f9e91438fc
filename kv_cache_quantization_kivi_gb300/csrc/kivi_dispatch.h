// kivi_dispatch.h -- selects the kernel instance for (bits, group, head_dim).
// head_dim 128 (every model shape these kernels are tuned for) has its own
// instances with compile-time address arithmetic; any other supported
// head_dim runs the generic instances (DC = 0, head_dim read at run time).
#pragma once

#define KIVI_DISPATCH_D(FN, B, G, P, STREAM) \
  return (P).d == 128 ? FN<B, G, 128>(P, STREAM) : FN<B, G, 0>(P, STREAM)

#define KIVI_DISPATCH(FN, P, GROUP, BITS, STREAM)                     \
  do {                                                                \
    switch ((BITS) * 1000 + (GROUP)) {                                \
      case 2016: KIVI_DISPATCH_D(FN, 2, 16, P, STREAM);               \
      case 4016: KIVI_DISPATCH_D(FN, 4, 16, P, STREAM);               \
      case 8016: KIVI_DISPATCH_D(FN, 8, 16, P, STREAM);               \
      case 2032: KIVI_DISPATCH_D(FN, 2, 32, P, STREAM);               \
      case 2064: KIVI_DISPATCH_D(FN, 2, 64, P, STREAM);               \
      case 2128: KIVI_DISPATCH_D(FN, 2, 128, P, STREAM);              \
      case 4032: KIVI_DISPATCH_D(FN, 4, 32, P, STREAM);               \
      case 4064: KIVI_DISPATCH_D(FN, 4, 64, P, STREAM);               \
      case 4128: KIVI_DISPATCH_D(FN, 4, 128, P, STREAM);              \
      case 8032: KIVI_DISPATCH_D(FN, 8, 32, P, STREAM);               \
      case 8064: KIVI_DISPATCH_D(FN, 8, 64, P, STREAM);               \
      case 8128: KIVI_DISPATCH_D(FN, 8, 128, P, STREAM);              \
      default: return cudaErrorInvalidValue;                          \
    }                                                                 \
  } while (0)

// The same for kernels with a compile-time mode M (see kivi_launch.h).
#define KIVI_DISPATCH_DM(FN, B, G, M, P, STREAM) \
  return (P).d == 128 ? FN<B, G, 128, M>(P, STREAM) : FN<B, G, 0, M>(P, STREAM)

#define KIVI_DISPATCH_BG(FN, P, GROUP, BITS, M, STREAM)                                  \
  switch ((BITS) * 1000 + (GROUP)) {                                                    \
    case 2016: KIVI_DISPATCH_DM(FN, 2, 16, M, P, STREAM);                               \
    case 4016: KIVI_DISPATCH_DM(FN, 4, 16, M, P, STREAM);                               \
    case 8016: KIVI_DISPATCH_DM(FN, 8, 16, M, P, STREAM);                               \
    case 2032: KIVI_DISPATCH_DM(FN, 2, 32, M, P, STREAM);                               \
    case 2064: KIVI_DISPATCH_DM(FN, 2, 64, M, P, STREAM);                               \
    case 2128: KIVI_DISPATCH_DM(FN, 2, 128, M, P, STREAM);                              \
    case 4032: KIVI_DISPATCH_DM(FN, 4, 32, M, P, STREAM);                               \
    case 4064: KIVI_DISPATCH_DM(FN, 4, 64, M, P, STREAM);                               \
    case 4128: KIVI_DISPATCH_DM(FN, 4, 128, M, P, STREAM);                              \
    case 8032: KIVI_DISPATCH_DM(FN, 8, 32, M, P, STREAM);                               \
    case 8064: KIVI_DISPATCH_DM(FN, 8, 64, M, P, STREAM);                               \
    case 8128: KIVI_DISPATCH_DM(FN, 8, 128, M, P, STREAM);                              \
    default: return cudaErrorInvalidValue;                                              \
  }

#define KIVI_DISPATCH_MODE(FN, P, GROUP, BITS, MODE, STREAM)                            \
  do {                                                                                  \
    switch (MODE) {                                                                     \
      case 0: KIVI_DISPATCH_BG(FN, P, GROUP, BITS, 0, STREAM)                           \
      case 1: KIVI_DISPATCH_BG(FN, P, GROUP, BITS, 1, STREAM)                           \
      case 2: KIVI_DISPATCH_BG(FN, P, GROUP, BITS, 2, STREAM)                           \
      default: return cudaErrorInvalidValue;                                            \
    }                                                                                   \
  } while (0)
