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
