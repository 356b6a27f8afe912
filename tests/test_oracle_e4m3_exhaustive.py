"""The oracle's E4M3 encoder on all 2^32 binary32 bit patterns, in C on every
host core: NaN gives 0x7F; every other input a finite code with the input's
sign; |x| >= 448 and infinities saturate to +-448; below that the code is a
nearest value with exact ties on the even code; codes never decrease as x
grows; code(-x) = code(x) | 0x80; and decoding then encoding returns every
finite code ("Engines for the card you have", "One checkpoint, many
engines": the FP8 key/value cache; OCP E4M3).  The checks are in
tests/e4m3_exhaustive.c, compiled here with oracle/oracle.c."""
import ctypes
import os
import subprocess

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
CHECKS = ["NaN -> 0x7F", "finite code with the input's sign", "saturation to +-448", "nearest value",
          "ties to even", "monotone", "symmetric in the sign", "decode -> encode identity"]


def test_e4m3_encoder_on_every_binary32_pattern(tmp_path):
    so = str(tmp_path / "e4m3_exhaustive.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math", "-pthread",
                    os.path.join(os.path.dirname(HERE), "oracle", "oracle.c"), os.path.join(HERE, "e4m3_exhaustive.c"),
                    "-o", so, "-lm"], check=True)
    lib = ctypes.CDLL(so)
    n = len(CHECKS)
    bad = (ctypes.c_uint64 * n)()
    first = (ctypes.c_uint32 * n)()
    lib.e4m3_exhaustive.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    lib.e4m3_exhaustive.restype = None
    lib.e4m3_exhaustive(oracle.host_cores(), ctypes.addressof(bad), ctypes.addressof(first))
    failed = {CHECKS[k]: (int(bad[k]), hex(first[k])) for k in range(n) if bad[k]}
    assert not failed, f"patterns failing (count, first pattern): {failed}"
