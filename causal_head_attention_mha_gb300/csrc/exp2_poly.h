// exp2_poly.h — written by gen_exp2_poly.py; do not edit.
// Minimax (Remez, relative error) polynomial of degree 3 for 2^f, f in [-1/2, 1/2].
// Max relative error in exact arithmetic: 7.478e-05.
#pragma once
#define MHA_EXP2_POLY_DEGREE 3
#define MHA_EXP2_POLY_C0 0.9999280571937561f
#define MHA_EXP2_POLY_C1 0.6932609677314758f
#define MHA_EXP2_POLY_C2 0.2426111251115799f
#define MHA_EXP2_POLY_C3 0.0551716685295105f
