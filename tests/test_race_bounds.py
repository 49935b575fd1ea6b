"""The bounds the race kernels prune with, checked on the host for every
value the uniform map can take (CPU only).

U = ((w >> 9) + 1/2) * 2^-23 takes 2^23 values.  With E = -ln U:
  * 1 - U <= E, so a key r / E never exceeds r / (1 - U): an entry whose
    r / (1 - U) does not beat the threshold cannot win;
  * E <= (1 - U) / U, so r U / (1 - U) never exceeds the key: the kernels
    seed their thresholds with r U / (1 - U) * (1 - 2^-18), and that margin
    must stay well above fp32 rounding (a few units of 2^-24) so a seed
    never exceeds the computed key of the entry it came from.
"""
import numpy as np


def _all_uniforms():
    k = np.arange(1 << 23, dtype=np.float64)
    return (k + 0.5) * 2.0**-23


def test_upper_bound_one_minus_u():
    U = _all_uniforms()
    E = -np.log(U)
    assert (E >= 1.0 - U).all()


def test_seed_lower_bound_keeps_a_margin_above_rounding():
    U = _all_uniforms()
    E = -np.log(U)
    seed = U / (1.0 - U) * (1.0 - 2.0**-18)  # per unit weight
    key = 1.0 / E
    # relative slack of the seed under the key: at least 2^-19, i.e. far
    # more than the few fp32 units of 2^-24 by which either side can round
    assert (seed <= key * (1.0 - 2.0**-19)).all()
    # without the shrink factor the slack near U = 1 is below fp32 resolution
    bare = U / (1.0 - U)
    assert ((key - bare) / key).min() < 2.0**-24


def test_fp32_one_minus_u_from_complemented_bits_is_exact():
    """The race kernels form 1 - U in fp32 as the float whose bits are
    (w >> 9) ^ 0x3FFFFFFF (the complemented 23 bits under the exponent of
    1.0) minus 1 - 2^-24.  Every one of the 2^23 values must come out
    exactly 1 - U: an overstated 1 - U makes the pruning bound r / (1 - U)
    too small and drops winners whose U lies within a few ulp of 1."""
    k = np.arange(1 << 23, dtype=np.uint32)
    one_minus_u = 1.0 - (k.astype(np.float64) + 0.5) * 2.0**-23
    f = ((k ^ np.uint32(0x7FFFFF)) | np.uint32(0x3F800000)).view(np.float32)
    y = f - np.float32(1.0 - 2.0**-24)
    assert y.dtype == np.float32
    assert (y.astype(np.float64) == one_minus_u).all()
    # and the fp32 value U itself, as the key's logarithm takes it
    u = (k | np.uint32(0x3F800000)).view(np.float32) - np.float32(1.0 - 2.0**-24)
    assert (u.astype(np.float64) == 1.0 - one_minus_u).all()
    assert (np.float32(1.0) - y == u).all()


def test_two_minus_half_ulp_is_not_an_fp32_number():
    """2 - 2^-24 lies halfway between two fp32 numbers and rounds (to even)
    to 2: a difference taken from it overstates 1 - U by 2^-24, which is
    the whole of 1 - U for the largest word."""
    assert np.float32(1.99999994039535522461) == np.float32(2.0)
    assert np.float32(1.0 - 2.0**-24) != np.float32(1.0)
