// fpd_grid.cu — f4: committed fixed-width numeral blocks -> the target's text format (host code only).
//
// VFlash paper (zh) §2.3: a coordinate of a text-tokenised target is drafted as one sign slot and `width` digit
// slots whose unused high digits hold the mask token; the grid is converted back to the target's text format.
// The layout and the text rule are stated with fpd_grid_to_text in include/fpd.h.
#include <cstdio>
#include <cstring>
#include <string>

#include "fpd_internal.cuh"

namespace fpd {
fpd_status set_last_error(fpd_status s, const char* msg);
}

namespace {

// Value of one field [sign][d_1..d_width] starting at tok, or false when the field breaks the schema.
bool field_value(const int32_t* tok, const fpd_grid_format& f, long long* value) {
  const bool neg = tok[0] == f.minus_id;
  if (!neg && tok[0] != f.plus_id) return false;
  long long v = 0;
  bool real = false;   // a real digit has been read: no pad may follow
  for (int i = 1; i <= f.width; i++) {
    const int32_t t = tok[i];
    if (t == f.pad_id) {
      if (real || i == f.width) return false;
      continue;
    }
    int d = -1;
    for (int k = 0; k < 10; k++)
      if (f.digit_id[k] == t) d = k;
    if (d < 0) return false;
    real = true;
    v = v * 10 + d;
  }
  *value = neg ? -v : v;
  return true;
}

}  // namespace

extern "C" fpd_status fpd_grid_to_text(int batch, int block_len, const int32_t* committed, const int32_t* accept,
                                       const fpd_grid_format* fmt, char* out, size_t out_bytes, size_t* offsets) {
  using fpd::set_last_error;
  if (batch < 1 || block_len < 2) return set_last_error(FPD_ERR_SHAPE, "batch < 1 or block_len < 2");
  if (!committed || !accept || !fmt || !out || !offsets) return set_last_error(FPD_ERR_INVALID_ARG, "null pointer argument");
  const fpd_grid_format& f = *fmt;
  if (f.n_axes < 1 || f.width < 1 || f.width > 18) return set_last_error(FPD_ERR_SHAPE, "n_axes >= 1 and 1 <= width <= 18");
  const int field = 1 + f.width, per_wp = f.n_axes * field + 1;
  size_t pos = 0;
  std::string text;
  for (int b = 0; b < batch; b++) {
    const int32_t* cm = committed + (size_t)b * block_len;   // cm[i] = block position i + 1
    int acc = accept[b];
    acc = acc < 0 ? 0 : (acc > block_len - 1 ? block_len - 1 : acc);
    text.clear();
    bool ok = true;
    for (int w = 0; ok; w++) {
      const int first = 1 + w * per_wp;                       // block position of the waypoint's first field
      if (first + f.n_axes * field - 1 > acc) break;         // not every field accepted
      std::string pt;
      for (int a = 0; a < f.n_axes; a++) {
        long long v = 0;
        if (!field_value(cm + first - 1 + a * field, f, &v)) {
          ok = false;
          break;
        }
        if (a) pt += f.axis_sep;
        pt += std::to_string(v);
      }
      if (!ok) break;
      if (w) text += f.point_sep;
      text += pt;
    }
    offsets[b] = pos;
    if (pos + text.size() + 1 > out_bytes) {
      offsets[batch] = pos + text.size() + 1;
      return set_last_error(FPD_ERR_CAPACITY, "text buffer too small");
    }
    memcpy(out + pos, text.c_str(), text.size() + 1);
    pos += text.size() + 1;
  }
  offsets[batch] = pos;
  return FPD_OK;
}
