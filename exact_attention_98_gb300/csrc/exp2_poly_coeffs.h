// Written by fit_exp2_poly.py -- do not edit by hand.
// 2^f ~ 1 + c1 f + ... + c3 f^3 on f in [-1/2, 1/2];
// minimax relative error 1.013e-04 (exact arithmetic), 1.013e-04 (fp32 Horner).
#pragma once
#define FA_EXP2_POLY_DEGREE 3
#define FA_EXP2_POLY_C1 0.6932829022407532f
#define FA_EXP2_POLY_C2 0.24221095442771912f
#define FA_EXP2_POLY_C3 0.05500892922282219f
#define FA_EXP2_POLY_MAX_REL_ERR 1.013448e-04
