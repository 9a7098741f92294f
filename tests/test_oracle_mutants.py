"""Plant plausible mistakes in a COPY of the oracle source (on the CPU) and check that
the pins in test_oracle_pins.py catch every one of them.

Each mutant is the oracle's C source with one textual change: a dropped term, a wrong
sign, a wrong index, a transposed operand, an off-by-one in a mask.  An anchor that
occurs in both the forward and the backward gives one mutant per occurrence.  A mutant that no
pin rejects would mean the pins leave that part of the oracle unchecked.
"""
import os
import tempfile

import pytest

from oracle import oracle as orc
import test_oracle_pins as pins

MUTANTS = {
    "tail_mask_off_by_one": ("(j % block) >= valid", "(j % block) > valid"),
    "lse_natural_log": ("lse[t * block + r] = (m + log(l)) / log(2.0);",
                        "lse[t * block + r] = m + log(l);"),
    "score_reads_query_row_of_k": ("bf16_to_double(kh[(int64_t)j * D + d])",
                                   "bf16_to_double(kh[(int64_t)i * D + d])"),
    "no_normalisation": ("orow[d] = acc[d] / l;", "orow[d] = acc[d];"),
    "exp_sign": ("const double p = exp(s_buf[a] - m);", "const double p = exp(m - s_buf[a]);"),
    "scale_dropped": ("s_buf[n_att] = scale * dot;", "s_buf[n_att] = dot;"),
    "count_not_clamped_reads_padding": ("for (int s = 0; s < n; ++s) {",
                                        "for (int s = 0; s < max_kv; ++s) {"),
    "range_check_dropped": ("if (kb >= 0 && kb < nb) mrow[kb] = 1;",
                            "if (kb >= 0 && kb < nb) mrow[kb] = 1; else if (kb >= 0) mrow[kb % nb] = 1;"),
    "mask_strides_swapped": ("(b * mask_stride_b + h * mask_stride_h)",
                             "(b * mask_stride_h + h * mask_stride_b)"),
    "v_row_from_query": ("vh + (int64_t)j_buf[a] * D", "vh + (int64_t)i * D"),
    "empty_row_lse_zero": ("lse[t * block + r] = ORACLE_LSE_EMPTY;", "lse[t * block + r] = 0.0;"),
    "lut_padding_zero": ("for (int s = n; s < max_kv; ++s) irow[s] = -1;",
                         "for (int s = n; s < max_kv; ++s) irow[s] = 0;"),
    "lut_descending": ("for (int kb = 0; kb < nb; ++kb) {\n      if (mrow[kb] != 0) {",
                       "for (int kb = nb - 1; kb >= 0; --kb) {\n      if (mrow[kb] != 0) {"),
    "bitmap_byte_must_be_one": ("if (mrow[kb] != 0) {", "if (mrow[kb] == 1) {"),
    "kv_head_interleaved": ("(int64_t)b * Hkv + h / group;", "(int64_t)b * Hkv + h % Hkv;"),
    "kv_head_stride_query_length": (
        "const uint16_t *kh = k + bkv * Sk * (int64_t)D;\n      const uint16_t *vh = v + bkv * Sk * (int64_t)D;\n      const int8_t",
        "const uint16_t *kh = k + bkv * Sq * (int64_t)D;\n      const uint16_t *vh = v + bkv * Sk * (int64_t)D;\n      const int8_t"),
    "bwd_kv_group_of_first_head": ("for (int h = hk * group; h < (hk + 1) * group; ++h) {",
                                   "for (int h = hk; h < hk + 1; ++h) {"),
    "mask_row_stride_query_blocks": ("(int64_t)qb * nbk;", "(int64_t)qb * nbq;"),
    "bwd_no_row_term": ("const double ds = p * (dp_buf[a] - Di);",
                        "const double ds = p * dp_buf[a];"),
    "bwd_dv_from_ds": ("dvh[j * D + d] += p * drow[d];", "dvh[j * D + d] += ds * drow[d];"),
    "bwd_dq_scale_dropped": ("dqh[(int64_t)i * D + d] += scale * ds * kd;",
                             "dqh[(int64_t)i * D + d] += ds * kd;"),
    "bwd_dk_from_dout": ("dkh[j * D + d] += scale * ds * qrow[d];",
                         "dkh[j * D + d] += scale * ds * drow[d];"),
    "bwd_dp_from_k": ("dpd += drow[d] * bf16_to_double(vh[(int64_t)j * D + d]);",
                      "dpd += drow[d] * bf16_to_double(kh[(int64_t)j * D + d]);"),
}


def _cases():
    """One mutant per occurrence of each anchor: the forward and the backward repeat some
    lines (the token mask, the score), and a slip in either copy must be caught."""
    src = open(orc.SRC).read()
    out = []
    for name in sorted(MUTANTS):
        n = src.count(MUTANTS[name][0])
        assert n >= 1, "mutation anchor missing: " + name
        out += [(name, i) for i in range(n)]
    return out


@pytest.mark.parametrize("name,occ", _cases(), ids=lambda x: str(x))
def test_pins_reject_mutant(name, occ):
    src = open(orc.SRC).read()
    old, new = MUTANTS[name]
    pos = -1
    for _ in range(occ + 1):
        pos = src.index(old, pos + 1)
    with tempfile.TemporaryDirectory() as d:
        msrc = os.path.join(d, "mutant.c")
        open(msrc, "w").write(src[:pos] + new + src[pos + len(old):])
        lib = orc.build(msrc, os.path.join(d, "libmutant.so"), openmp=False)
        h = orc.load(lib, msrc)
        caught = []
        for pin in pins.PINS:
            try:
                pin(h)
            except AssertionError:
                caught.append(pin.__name__)
        assert caught, "no pin rejects mutant %s (occurrence %d)" % (name, occ)
