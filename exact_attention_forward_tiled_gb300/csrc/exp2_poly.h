// Written by exp2_poly_fit.py -- do not edit by hand.
// 2^f on [-1/2, 1/2] by a degree-3 minimax (relative error) polynomial,
// Remez exchange in float64; max relative error 7.478e-05 (float64 coefficients),
// 7.483e-05 with these fp32 coefficients evaluated in fp32 Horner form.
#pragma once
namespace fa {
constexpr float kExp2C0 = 0.9999280571937561f;
constexpr float kExp2C1 = 0.6932609677314758f;
constexpr float kExp2C2 = 0.2426111251115799f;
constexpr float kExp2C3 = 0.0551716685295105f;
}  // namespace fa
