// hl_tanh_poly.h -- written by fit_tanh_poly.py; do not edit.
// tanh(y) ~= y * P(y^2) for |y| <= Y0, P(0) = 1 (coefficients C0 .. Cdeg).
#pragma once
// HL_TANH_POLY: degree 6 on |y| <= 0.8; max relative error of the real-valued fit 3.34e-09
#define HL_TANH_POLY_Y0 0.8f
#define HL_TANH_POLY_C0 1.0f
#define HL_TANH_POLY_C1 -0.3333328068256378f
#define HL_TANH_POLY_C2 0.13332021236419678f
#define HL_TANH_POLY_C3 -0.053841542452573776f
#define HL_TANH_POLY_C4 0.02127472497522831f
#define HL_TANH_POLY_C5 -0.007374097593128681f
#define HL_TANH_POLY_C6 0.0015676695620641112f
// HL_TANH_A: degree 3 on |y| <= 0.45; max relative error of the real-valued fit 2.44e-07
#define HL_TANH_A_Y0 0.45f
#define HL_TANH_A_C0 1.0f
#define HL_TANH_A_C1 -0.33329465985298157f
#define HL_TANH_A_C2 0.13236358761787415f
#define HL_TANH_A_C3 -0.04602816700935364f
// HL_TANH_B: degree 5 on |y| <= 0.8; max relative error of the real-valued fit 5.81e-08
#define HL_TANH_B_Y0 0.8f
#define HL_TANH_B_C0 1.0f
#define HL_TANH_B_C1 -0.3333267569541931f
#define HL_TANH_B_C2 0.1332104504108429f
#define HL_TANH_B_C3 -0.05311424657702446f
#define HL_TANH_B_C4 0.019093237817287445f
#define HL_TANH_B_C5 -0.004355288110673428f
