"""Philox4x64-10 counter-based generator in vectorised numpy.

Definition (Salmon et al., SC'11, the Philox family): a 4x64-bit counter and
a 2x64-bit key; each of 10 rounds multiplies counter words 0 and 2 by two
fixed odd constants, producing 128-bit products whose high halves are
xored with the other two counter words and the key, and the key is bumped
by two Weyl constants between rounds.  numpy's ``np.random.Philox`` is the
same function, which the tests use as an independent pin.

The device twin lives in ``synth/csrc/synth_dev.cu``.
"""

import numpy as np

_M0 = np.uint64(0xD2E7470EE14C6C93)
_M1 = np.uint64(0xCA5A826395121157)
_W0 = np.uint64(0x9E3779B97F4A7C15)
_W1 = np.uint64(0xBB67AE8584CAA73B)
_LO32 = np.uint64(0xFFFFFFFF)
_S32 = np.uint64(32)


def _mulhilo(a, b):
    """128-bit product of uint64 arrays, returned as (hi, lo)."""
    a = np.asarray(a, dtype=np.uint64)
    b = np.asarray(b, dtype=np.uint64)
    al, ah = a & _LO32, a >> _S32
    bl, bh = b & _LO32, b >> _S32
    t = al * bl
    w0 = t & _LO32
    k = t >> _S32
    t = ah * bl + k
    w1 = t & _LO32
    w2 = t >> _S32
    t = al * bh + w1
    k = t >> _S32
    hi = ah * bh + w2 + k
    lo = (t << _S32) | w0
    return hi, lo


def philox4x64(c0, c1, c2, c3, k0, k1):
    """Philox4x64-10 of counter (c0..c3) under key (k0, k1).

    All arguments broadcast as uint64 arrays.  Returns a uint64 array of
    shape ``broadcast_shape + (4,)``.
    """
    with np.errstate(over="ignore"):
        c0, c1, c2, c3, k0, k1 = np.broadcast_arrays(
            *(np.asarray(x, dtype=np.uint64) for x in (c0, c1, c2, c3, k0, k1))
        )
        c0, c1, c2, c3 = c0.copy(), c1.copy(), c2.copy(), c3.copy()
        k0, k1 = k0.copy(), k1.copy()
        for _ in range(10):
            hi0, lo0 = _mulhilo(_M0, c0)
            hi1, lo1 = _mulhilo(_M1, c2)
            c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
            k0 = k0 + _W0
            k1 = k1 + _W1
        return np.stack([c0, c1, c2, c3], axis=-1)


def philox_u32(stream_key0, stream_key1, flat_index):
    """The 32-bit word number ``flat_index`` of one Philox stream.

    A stream is the key (k0, k1); word i is taken from the output of
    counter (i // 8, 0, 0, 0): output word w = (i % 8) // 2, low half for
    even i and high half for odd i.  ``flat_index`` is a uint64 array.
    """
    i = np.asarray(flat_index, dtype=np.uint64)
    blk = i >> np.uint64(3)
    sub = (i & np.uint64(7)).astype(np.int64)
    out = philox4x64(blk, 0, 0, 0, stream_key0, stream_key1)
    word = np.take_along_axis(out, (sub // 2)[..., None], axis=-1)[..., 0]
    shift = (sub % 2).astype(np.uint64) * _S32
    return ((word >> shift) & _LO32).astype(np.uint32)
