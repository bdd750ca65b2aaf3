"""Pins for the oracle's counter-based generator (Philox4x32-10, Salmon et al., SC'11).

The pages name Philox as the noise source (Megatron-LM PR "The change"; spec-decode-ops
"Randomness is counter-based Philox") but print no known-answer vectors.  The pin used here is
a second, independent implementation that is *run*, not retyped: Triton's ``tl.philox``
executed by Triton's CPU interpreter, over 10^4 random (key, counter) pairs, the corner values,
and several round counts (which also pins the key schedule between rounds).
"""
import json
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_TRITON_SCRIPT = textwrap.dedent(r"""
    import os, sys, json
    os.environ["TRITON_INTERPRET"] = "1"
    import numpy as np, torch, triton, triton.language as tl

    @triton.jit
    def kern(out, k0p, k1p, c0p, c1p, c2p, c3p, N: tl.constexpr, R: tl.constexpr):
        i = tl.arange(0, N)
        k0 = tl.load(k0p + i).to(tl.uint32).to(tl.uint64)
        k1 = tl.load(k1p + i).to(tl.uint32).to(tl.uint64)
        seed = (k1 << 32) | k0
        c0 = tl.load(c0p + i); c1 = tl.load(c1p + i); c2 = tl.load(c2p + i); c3 = tl.load(c3p + i)
        a, b, c, d = tl.philox(seed, c0, c1, c2, c3, R)
        tl.store(out + i * 4 + 0, a); tl.store(out + i * 4 + 1, b)
        tl.store(out + i * 4 + 2, c); tl.store(out + i * 4 + 3, d)

    data = np.load(sys.argv[1])
    ctr, key, rounds = data["ctr"], data["key"], int(data["rounds"])
    n = ctr.shape[0]
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int32))
    out = torch.zeros(n * 4, dtype=torch.int32)
    kern[(1,)](out, t(key[:, 0]), t(key[:, 1]), t(ctr[:, 0]), t(ctr[:, 1]), t(ctr[:, 2]),
               t(ctr[:, 3]), N=n, R=rounds)
    np.save(sys.argv[2], out.numpy().view(np.uint32).reshape(n, 4))
""")


def _triton_philox(ctr, key, rounds, tmp_path):
    pytest.importorskip("triton")
    pytest.importorskip("torch")
    inp = tmp_path / f"in_{rounds}.npz"
    outp = tmp_path / f"out_{rounds}.npy"
    np.savez(inp, ctr=ctr, key=key, rounds=rounds)
    script = tmp_path / "tri.py"
    script.write_text(_TRITON_SCRIPT)
    env = dict(os.environ, TRITON_INTERPRET="1")
    r = subprocess.run([sys.executable, str(script), str(inp), str(outp)], env=env,
                       capture_output=True, text=True, timeout=600)
    if r.returncode != 0:
        pytest.skip(f"Triton interpreter unavailable: {r.stderr[-400:]}")
    return np.load(outp)


def _cases(n, seed):
    rng = np.random.default_rng(seed)
    ctr = rng.integers(0, 2**32, size=(n, 4), dtype=np.uint64).astype(np.uint32)
    key = rng.integers(0, 2**32, size=(n, 2), dtype=np.uint64).astype(np.uint32)
    edge = np.array([0, 1, 0x7FFFFFFF, 0x80000000, 0xFFFFFFFF], dtype=np.uint32)
    ce = np.array(np.meshgrid(edge, edge, indexing="ij")).reshape(2, -1).T
    ctr[: len(ce), 0] = ce[:, 0]
    ctr[: len(ce), 3] = ce[:, 1]
    key[: len(ce), 0] = ce[:, 1]
    key[: len(ce), 1] = ce[:, 0]
    ctr[len(ce)] = 0
    key[len(ce)] = 0
    ctr[len(ce) + 1] = 0xFFFFFFFF
    key[len(ce) + 1] = 0xFFFFFFFF
    return ctr, key


def test_philox4x32_10_matches_triton_interpreter(tmp_path):
    ctr, key = _cases(16384, 1)
    ours = oracle.philox4x32(ctr, key, 10)
    theirs = _triton_philox(ctr, key, 10, tmp_path)
    assert ours.dtype == np.uint32 and theirs.shape == ours.shape
    bad = np.nonzero((ours != theirs).any(axis=1))[0]
    assert bad.size == 0, f"{bad.size} mismatches, first ctr={ctr[bad[0]]} key={key[bad[0]]}"


@pytest.mark.parametrize("rounds", [1, 2, 7])
def test_philox_round_counts_match_triton(tmp_path, rounds):
    # Fewer rounds expose the round function and the per-round key bump separately.
    ctr, key = _cases(1024, 2 + rounds)
    assert (oracle.philox4x32(ctr, key, rounds) == _triton_philox(ctr, key, rounds, tmp_path)).all()


def test_philox_zero_rounds_is_identity():
    ctr, key = _cases(64, 9)
    assert (oracle.philox4x32(ctr, key, 0) == ctr).all()


def test_philox_output_bits_are_balanced():
    # 2^18 outputs of consecutive counters: every one of the 128 output bits is set about half
    # the time (a dropped round or a swapped word leaves strong bias in low-round outputs).
    n = 1 << 18
    ctr = np.zeros((n, 4), np.uint32)
    ctr[:, 0] = np.arange(n, dtype=np.uint32)
    key = np.tile(np.array([1234, 0], np.uint32), (n, 1))
    out = oracle.philox4x32(ctr, key, 10)
    bits = np.unpackbits(out.view(np.uint8), axis=1)
    frac = bits.mean(axis=0)
    assert np.all(np.abs(frac - 0.5) < 6 * 0.5 / np.sqrt(n))


def test_seeded_key_counter_is_injective_and_disjoint_from_unseeded():
    # (seed, position, v) -> (key, counter) must be injective, and seeded counters never
    # collide with unseeded ones (their fourth word carries the top bit).
    from itertools import product
    seen = set()
    import ctypes
    lib = oracle._load()
    lib.orc_key_counter.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_uint64,
                                    ctypes.c_uint64, ctypes.c_int64, ctypes.c_uint32,
                                    ctypes.c_void_p, ctypes.c_void_p]
    ctr = np.zeros(4, np.uint32)
    key = np.zeros(2, np.uint32)
    for seeded, a, p, v in product([0, 1], [0, 1, 2**32, 2**40 + 3], [0, 1, 2**32, 5 * 2**33], [0, 1, 151935]):
        if seeded:
            lib.orc_key_counter(1, a, p, 0, 0, 0, v, oracle._ptr(ctr), oracle._ptr(key))
        else:
            lib.orc_key_counter(0, -1, 0, a, p, 7, v, oracle._ptr(ctr), oracle._ptr(key))
        t = tuple(ctr.tolist() + key.tolist())
        assert t not in seen
        seen.add(t)
        assert bool(ctr[3] & 0x80000000) == (not seeded)
