"""Writes rng_vectors.txt: (seed, b, pos, stream, v) -> the splitmix64 hash of
key ^ (v >> 1) (one hash serves entries 2j and 2j + 1) and the uniform of entry
v, computed by the CPU oracle only.  The GPU tests compare the CUDA
library's generator against these lines bit for bit.

    python tests/golden/make_rng_vectors.py
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402

CASES = [
    (0, 0, 0, 0, 0), (0, 0, 0, 1, 0), (0, 0, 0, 1, 1), (0, 1, 0, 0, 0), (0, 0, 1, 0, 0),
    (1, 0, 0, 0, 0), (4, 1023, 7, 1, 255999), (3, 255, 8, 1, 151935), (2, 63, 7, 0, 0),
    (0xFFFFFFFFFFFFFFFF, 5, 3, 1, 77), (123456789, 42, 31, 1, 1 << 20), (7, 1 << 30, 100, 0, 0),
    (4, 1023, 7, 1, 255998), (0xFFFFFFFFFFFFFFFF, 5, 3, 1, 76), (0, 0, 0, 0, 1),
]


def main():
    path = os.path.join(HERE, "rng_vectors.txt")
    with open(path, "w") as f:
        f.write("# seed b pos stream v  splitmix64(key ^ (v >> 1))  U\n")
        f.write("# written by tests/golden/make_rng_vectors.py from the CPU oracle\n")
        for seed, b, pos, stream, v in CASES:
            h = oracle.splitmix64(oracle.stream_key(seed, b, pos, stream) ^ (v >> 1))
            u = oracle.uniform(seed, b, pos, stream, v, 1)[0]
            f.write(f"{seed:#x} {b} {pos} {stream} {v} {h:016x} {float(u).hex()}\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
