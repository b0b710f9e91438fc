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

// The same for kernels with a compile-time reconstruction flag R.
#define KIVI_DISPATCH_DR(FN, B, G, R, P, STREAM) \
  return (P).d == 128 ? FN<B, G, 128, R>(P, STREAM) : FN<B, G, 0, R>(P, STREAM)

#define KIVI_DISPATCH_R(FN, P, GROUP, BITS, RECON, STREAM)                              \
  do {                                                                                  \
    if (RECON) {                                                                        \
      switch ((BITS) * 1000 + (GROUP)) {                                                \
        case 2032: KIVI_DISPATCH_DR(FN, 2, 32, true, P, STREAM);                        \
        case 2064: KIVI_DISPATCH_DR(FN, 2, 64, true, P, STREAM);                        \
        case 2128: KIVI_DISPATCH_DR(FN, 2, 128, true, P, STREAM);                       \
        case 4032: KIVI_DISPATCH_DR(FN, 4, 32, true, P, STREAM);                        \
        case 4064: KIVI_DISPATCH_DR(FN, 4, 64, true, P, STREAM);                        \
        case 4128: KIVI_DISPATCH_DR(FN, 4, 128, true, P, STREAM);                       \
        case 8032: KIVI_DISPATCH_DR(FN, 8, 32, true, P, STREAM);                        \
        case 8064: KIVI_DISPATCH_DR(FN, 8, 64, true, P, STREAM);                        \
        case 8128: KIVI_DISPATCH_DR(FN, 8, 128, true, P, STREAM);                       \
        default: return cudaErrorInvalidValue;                                          \
      }                                                                                 \
    }                                                                                   \
    switch ((BITS) * 1000 + (GROUP)) {                                                  \
      case 2032: KIVI_DISPATCH_DR(FN, 2, 32, false, P, STREAM);                         \
      case 2064: KIVI_DISPATCH_DR(FN, 2, 64, false, P, STREAM);                         \
      case 2128: KIVI_DISPATCH_DR(FN, 2, 128, false, P, STREAM);                        \
      case 4032: KIVI_DISPATCH_DR(FN, 4, 32, false, P, STREAM);                         \
      case 4064: KIVI_DISPATCH_DR(FN, 4, 64, false, P, STREAM);                         \
      case 4128: KIVI_DISPATCH_DR(FN, 4, 128, false, P, STREAM);                        \
      case 8032: KIVI_DISPATCH_DR(FN, 8, 32, false, P, STREAM);                         \
      case 8064: KIVI_DISPATCH_DR(FN, 8, 64, false, P, STREAM);                         \
      case 8128: KIVI_DISPATCH_DR(FN, 8, 128, false, P, STREAM);                        \
      default: return cudaErrorInvalidValue;                                            \
    }                                                                                   \
  } while (0)
