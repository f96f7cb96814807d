// Drafter configuration from a checkpoint's config.json text, and the rotary-width rule
// ("memra_engine/eagle.rs", EagleConfig: from_json_str, rope_dim_count and the
// draft_rope_width_tests on the eagle3-qwen35-9b config).  Host code only.
//
// Keys are found the way the page's loader finds them: the first occurrence of the quoted
// key anywhere in the text, then the number after the colon.  A factor declared only under
// "rope_parameters" is therefore read as well as a top-level one, and rope_theta is read
// from wherever the config puts it.
#include <cmath>
#include <cstdlib>
#include <cstring>

#include "eagle3.h"

namespace {

// The number following "key": in json; false when the key is absent or its value is not a
// number (null, a string, an object).
bool json_number(const char *json, const char *key, double *out) {
  char pat[96];
  const size_t kl = std::strlen(key);
  if (kl + 3 > sizeof(pat)) return false;
  pat[0] = '"';
  std::memcpy(pat + 1, key, kl);
  pat[kl + 1] = '"';
  pat[kl + 2] = '\0';
  const char *at = std::strstr(json, pat);
  if (!at) return false;
  const char *p = at + kl + 2;
  while (*p == ' ' || *p == '\t' || *p == '\r' || *p == '\n') ++p;
  if (*p != ':') return false;
  ++p;
  while (*p == ' ' || *p == '\t' || *p == '\r' || *p == '\n') ++p;
  char *end = nullptr;
  const double v = std::strtod(p, &end);
  if (end == p) return false;
  while (*end == ' ' || *end == '\t' || *end == '\r') ++end;
  if (*end != ',' && *end != '}' && *end != '\n' && *end != '\0') return false;
  *out = v;
  return true;
}

bool json_int(const char *json, const char *key, int *out) {
  double v = 0.0;
  if (!json_number(json, key, &v)) return false;
  if (!(v >= 1.0 && v <= 2147483647.0) || std::floor(v) != v) return false;
  *out = (int)v;
  return true;
}

// A true / false value of "key"; -1 when absent or not a boolean.
int json_bool(const char *json, const char *key) {
  char pat[96];
  const size_t kl = std::strlen(key);
  if (kl + 3 > sizeof(pat)) return -1;
  pat[0] = '"';
  std::memcpy(pat + 1, key, kl);
  pat[kl + 1] = '"';
  pat[kl + 2] = '\0';
  const char *at = std::strstr(json, pat);
  if (!at) return -1;
  const char *p = at + kl + 2;
  while (*p == ' ' || *p == '\t' || *p == '\r' || *p == '\n') ++p;
  if (*p != ':') return -1;
  ++p;
  while (*p == ' ' || *p == '\t' || *p == '\r' || *p == '\n') ++p;
  if (std::strncmp(p, "true", 4) == 0) return 1;
  if (std::strncmp(p, "false", 5) == 0) return 0;
  return -1;
}

// Entries of the aux-layer id list ("eagle_aux_hidden_state_layer_ids": [1, 15, 28]);
// -1 when the key is absent, -2 when the list is malformed.
int aux_layer_count(const char *json) {
  const char *at = std::strstr(json, "\"eagle_aux_hidden_state_layer_ids\"");
  if (!at) return -1;
  const char *lb = std::strchr(at, '[');
  if (!lb) return -2;
  const char *rb = std::strchr(lb, ']');
  if (!rb) return -2;
  int n = 0;
  const char *p = lb + 1;
  while (p < rb) {
    char *end = nullptr;
    const long v = std::strtol(p, &end, 10);
    if (end == p) {
      ++p;
      continue;
    }
    if (v < 0) return -2;
    ++n;
    p = end;
  }
  return n;
}

}  // namespace

extern "C" int eagle3_resolve_rope_dims(int head_dim, int has_rotary_dim, int rotary_dim, int has_factor,
                                        float factor) {
  if (head_dim <= 0 || head_dim % 2) return 0;
  // an explicit count is the more specific declaration
  if (has_rotary_dim && rotary_dim >= 2 && rotary_dim <= head_dim && rotary_dim % 2 == 0) return rotary_dim;
  if (has_factor && factor > 0.f && factor <= 1.f) {
    const double d = (double)factor * head_dim;
    const double r = std::nearbyint(d);
    // a fraction that does not give a whole, even number of dims is malformed
    if (std::fabs(d - r) < 1e-6 && (long)r >= 2 && (long)r % 2 == 0) return (int)r;
  }
  return head_dim;  // no usable declaration: every head dim rotates
}

extern "C" int eagle3_config_from_json(const char *json, eagle3_config *cfg) {
  if (!json || !cfg) return EAGLE3_ERR_INVALID_ARG;
  eagle3_config c = *cfg;
  if (!json_int(json, "hidden_size", &c.n_embd) || !json_int(json, "num_attention_heads", &c.n_head) ||
      !json_int(json, "num_key_value_heads", &c.n_head_kv) || !json_int(json, "head_dim", &c.head_dim) ||
      !json_int(json, "intermediate_size", &c.n_ff) || !json_int(json, "draft_vocab_size", &c.draft_vocab) ||
      !json_int(json, "vocab_size", &c.target_vocab))
    return EAGLE3_ERR_INVALID_ARG;
  double v = 0.0;
  int has_rd = 0, rd = 0, has_f = 0;
  float f = 0.f;
  if (json_number(json, "rotary_dim", &v)) {
    has_rd = 1;
    rd = (v >= 0.0 && v <= 1e6 && std::floor(v) == v) ? (int)v : -1;
  }
  if (json_number(json, "partial_rotary_factor", &v)) {
    has_f = 1;
    f = (float)v;
  }
  c.rope_dims = eagle3_resolve_rope_dims(c.head_dim, has_rd, rd, has_f, f);
  c.rope_theta = json_number(json, "rope_theta", &v) ? (float)v : 10000.0f;
  c.rms_eps = json_number(json, "rms_norm_eps", &v) ? (float)v : 1e-6f;
  if (!(c.rope_theta > 0.f) || !(c.rms_eps >= 0.f)) return EAGLE3_ERR_INVALID_ARG;
  // checkpoint flags: only norm_before_residual is built; a config that turns on one of
  // the others is refused rather than run with the wrong op sequence
  c.flags = 0u;
  if (json_bool(json, "norm_before_residual") == 1) c.flags |= EAGLE3_CKPT_NORM_BEFORE_RESIDUAL;
  if (json_bool(json, "norm_before_fc") == 1 || json_bool(json, "fc_norm") == 1 ||
      json_bool(json, "norm_output") == 1)
    return EAGLE3_ERR_UNSUPPORTED;
  const int n_aux = aux_layer_count(json);
  if (n_aux == -2) return EAGLE3_ERR_INVALID_ARG;
  if (n_aux >= 0 && n_aux != 3) return EAGLE3_ERR_UNSUPPORTED;  // fc takes three features
  *cfg = c;
  return EAGLE3_OK;
}
