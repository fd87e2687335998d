"""Plant plausible mistakes in a copy of the oracle source (CPU only) and require every copy to
fail at least one pin.  This shows the pins constrain each stage of the oracle: the Haar filters,
the conv indexing, the scale pass, where the reconstruction enters the cascade, the base path and
each transpose of the backward."""
import os

import pytest

import oracle
import oracle_pins

# (name, original text, replacement): each original must occur exactly once in the source.
MUTANTS = [
    ("LH pattern made equal to HH", "{{1.0, -1.0}, {1.0, -1.0}}, /* LH */",
     "{{1.0, -1.0}, {-1.0, 1.0}}, /* LH */"),
    ("conv kernel transposed",
     "int r = i + u - p, c = j + v - p;\n                    if (r >= 0 && r < H && c >= 0 && c < W)\n                        acc += ker[u * k + v]",
     "int r = i + u - p, c = j + v - p;\n                    if (r >= 0 && r < H && c >= 0 && c < W)\n                        acc += ker[v * k + u]"),
    ("conv padding off by one", "void oracle_dwconv(const double *in, int H, int W, const double *ker, int k, double *out)\n{\n    int p = k / 2;",
     "void oracle_dwconv(const double *in, int H, int W, const double *ker, int k, double *out)\n{\n    int p = k / 2 + 1;"),
    ("every subband uses the LL scale",
     "double sc = J->wavelet_scale[(size_t)(l - 1) * 4 * C + 4 * c + sb];",
     "double sc = J->wavelet_scale[(size_t)(l - 1) * 4 * C + 4 * c];"),
    ("reconstruction added to LH instead of LL", "s->Z[l][i] += s->R[i]; /* subband 0 = LL */",
     "s->Z[l][h * w + i] += s->R[i];"),
    ("next level analyses LH instead of LL", "LL = s->Y[l]; /* subband 0 is the first [h_l][w_l] block */",
     "LL = s->Y[l] + (size_t)h * w;"),
    ("odd side padded at the start", "s->Pd[i * (2 * w) + j] = LL[i * wi + j];",
     "s->Pd[(i + 2 * h - hi) * (2 * w) + j + 2 * w - wi] = LL[i * wi + j];"),
    ("reconstruction cropped at the start", "s->R[i * wo + j] = s->R2[i * (2 * w) + j];",
     "s->R[i * wo + j] = s->R2[(i + 2 * h - ho) * (2 * w) + j + 2 * w - wo];"),
    ("backward: crop transpose pads at the start", "s->dR2[i * (2 * w) + j] = s->dR[i * wo + j];",
     "s->dR2[(i + 2 * h - ho) * (2 * w) + j + 2 * w - wo] = s->dR[i * wo + j];"),
    ("backward: pad transpose keeps the end", "s->dR2[i * wi + j] = s->Pd[i * (2 * w) + j];",
     "s->dR2[i * wi + j] = s->Pd[(i + 2 * h - hi) * (2 * w) + j + 2 * w - wi];"),
    ("base bias not scaled", "y[i] = sb_ * (s->base[i] + bb) + s->R[i];",
     "y[i] = sb_ * s->base[i] + bb + s->R[i];"),
    ("backward: base scale dropped from dbase", "s->dbase[i] = sb_ * dy[i];", "s->dbase[i] = dy[i];"),
    ("backward: bias grad not scaled", "g_base_bias[c] += sb_ * acc_bias;", "g_base_bias[c] += acc_bias;"),
    ("backward: kernel grad transposed", "d_ker[u * k + v] += in[r * W + c] * d_out[i * W + j];",
     "d_ker[v * k + u] += in[r * W + c] * d_out[i * W + j];"),
    ("backward: LL gradient from the next level dropped", "s->dY[l][i] += s->dR2[i];", "(void)0;"),
    ("backward: cascade gradient taken from LH", "memcpy(s->dR, s->dZ[l], (size_t)h * w * sizeof(double)); /* LL block */",
     "memcpy(s->dR, s->dZ[l] + (size_t)h * w, (size_t)h * w * sizeof(double));"),
    ("backward: scale grad uses scaled output", "acc += s->dZ[l][sb * n + i] * s->T[l][sb * n + i];",
     "acc += s->dZ[l][sb * n + i] * s->Z[l][sb * n + i];"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new, tmp_path):
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation site not unique / missing: {name}"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = oracle.compile_library(str(path), str(tmp_path / "libmutant.so"))
    orc = oracle.Oracle(lib)
    failures = []
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(orc)
        except (AssertionError, ValueError) as e:
            failures.append(f"{check.__name__}: {e}")
            break
    assert failures, f"mutant '{name}' passed every pin"
