// hl_tanh_poly.h -- written by fit_tanh_poly.py; do not edit.
// tanh(y) ~= y * P(y^2) for |y| <= 0.8; P of degree 6 in u = y^2, P(0) = 1.
// Max relative error of the real-valued fit: 3.34e-09.
#pragma once
#define HL_TANH_POLY_Y0 0.8f
#define HL_TANH_POLY_C0 1.0f
#define HL_TANH_POLY_C1 -0.3333328068256378f
#define HL_TANH_POLY_C2 0.13332021236419678f
#define HL_TANH_POLY_C3 -0.053841542452573776f
#define HL_TANH_POLY_C4 0.02127472497522831f
#define HL_TANH_POLY_C5 -0.007374097593128681f
#define HL_TANH_POLY_C6 0.0015676695620641112f
