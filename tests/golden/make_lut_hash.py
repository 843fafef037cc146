"""Writes tests/golden/mxfp4_half_lut.sha256: the SHA-256 of the oracle's 4096-entry MXFP4 -> half table
("quantization" glossary, "Metal MXFP4 -> half LUT": the generated table is pinned by its hash so that a change
of the generator shows up as drift). Calls only the oracle. Run: python tests/golden/make_lut_hash.py"""
import hashlib
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))
import oracle  # noqa: E402


def lut_sha256() -> str:
    lut = oracle.mxfp4_half_lut()  # [256 exponents][16 codes] uint16, row-major, little-endian bytes
    return hashlib.sha256(lut.astype("<u2").tobytes()).hexdigest()


if __name__ == "__main__":
    with open(os.path.join(HERE, "mxfp4_half_lut.sha256"), "w") as f:
        f.write(lut_sha256() + "\n")
