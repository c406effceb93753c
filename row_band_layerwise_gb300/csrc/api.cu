// C ABI of the decoder: weight repacking, workspace planning, and the layer walk
// that enqueues the kernels of one decode.
//
// The walk follows the decoder module order.  One GPU holds every band, so:
//  * convs run as one launch over all rows: a band's halo rows are its
//    neighbour's rows in the same tensor, read in place, and zero padding
//    appears only outside the image ("VAEP：VAE 并行解码", 卷积：交换边界行);
//  * GroupNorm statistics come from fixed one-row chunks merged with the
//    weighted rule (GroupNorm：合并全局统计量), independent of the band split;
//  * attention takes each band's query rows against every key and value of the
//    frame (Attention：本地 Q，全局 K/V): on the bf16 path one fused kernel covers
//    all bands, its query tiles never crossing a band, and no scores reach
//    memory; the fp32 path runs band by band with one band's scores in memory;
//  * SiLU, RMSNorm and upsampling are local (the upsample is folded into the
//    next conv's addressing).
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <map>
#include <sstream>
#include <string>
#include <vector>

#include "vaedec.h"
#include "kernels.h"

using namespace vd;

namespace {

thread_local std::string g_err;

vaedec_status fail(vaedec_status s, const std::string& m) {
  g_err = m;
  return s;
}

vaedec_status cuda_fail(cudaError_t e, const std::string& where) {
  return fail(VAEDEC_ERR_CUDA, where + ": " + cudaGetErrorString(e));
}

constexpr int kNumAct = 5;
constexpr size_t kSlotAlign = 256;          // every workspace slot starts on a 256-byte boundary
constexpr size_t kArenaGuard = 1 << 20;     // spare bytes after the last slot

// Process-wide failure injection (vaedec_debug_inject_fault).
std::atomic<int> g_fault_kind{0};
std::atomic<int> g_fault_left{0};

// True when the injected fault of `kind` fires now (it fires once, then switches off).
bool fault_now(int kind) {
  if (g_fault_kind.load() != kind) return false;
  if (g_fault_left.fetch_sub(1) == 1) {
    g_fault_kind.store(0);
    return true;
  }
  return false;
}

struct DevConv {
  void* w = nullptr;     // [rows][ntaps][cin] model dtype
  void* wup = nullptr;   // bf16 upsample convs: [rows][4 phases x 7][cin] two-by-two phase weights (hi, lo parts)
  void* wn = nullptr;    // bf16 3x3(x kt) convs with 3 outputs: [16][kt * 3][cin], row = kernel_row * 3 + co
  float* b_sc = nullptr; // a resnet conv2: its bias plus the block's shortcut bias (fused shortcut)
  float* b = nullptr;    // [cout]
  int rows = 0, ntaps = 0, cin = 0, cout = 0;
  int kt = 1, kh = 1, kw = 1;
};

struct DevNorm {
  float* g = nullptr;
  float* b = nullptr;
  int c = 0;
};

struct Act {
  int buf = -1;          // activation role index (>= 0: lives in the workspace arena), or -1 for an external pointer
  int slot = -1;         // workspace slot of an arena tensor (its offset comes from the liveness plan)
  void* ext = nullptr;
  int dt = kBF16;        // element type (kF32 / kBF16)
  int B = 0, T = 1, H = 0, W = 0, C = 0;
  // GroupNorm chunk moments written by the producing conv: chunks per sample and the
  // producer's sequence number (they are valid while no later conv overwrote them)
  int stats_chunks = 0;
  long long stats_epoch = -1;
  long long pixels() const { return (long long)B * T * H * W; }
};

enum ConvKind { K3, K1, C3, UP, TIME };

// Nearest-2x upsample then a 3x3 conv, output phase (py, px) on the low-resolution grid: the kernel
// rows i fall on low-resolution row offsets floor((py + i - 1) / 2), i.e. two offsets per phase,
// one taking a single kernel row and one the sum of two (likewise for columns).  So each phase is
// a two-by-two conv whose weights are sums of 1, 2, 2 and 4 of the 3x3 weights.  Those sums are
// not bf16 values; each is split into hi = bf16(sum) and lo = bf16(sum - hi), which together hold
// it to 2^-17 of its size, so the phase has 7 weight taps (the single weight needs no lo part)
// instead of the 9 taps of the direct form, with the same arithmetic up to that rounding.
struct UpTap {
  int oy, ox;            // low-resolution offsets
  int lo;                // 0: hi part of the summed weight, 1: lo part
  int nrow, ncol;        // kernel rows / columns summed
  int rows[2], cols[2];
};

constexpr int kUpTaps = 7;

void up_phase_taps(int ph, UpTap (&t)[kUpTaps]) {
  const int py = ph >> 1, px = ph & 1;
  // (offset, kernel indices) of the single-index and the two-index group along one axis
  struct Grp { int off, n, idx[2]; };
  const Grp ry1 = py == 0 ? Grp{-1, 1, {0, 0}} : Grp{1, 1, {2, 2}};
  const Grp ry2 = py == 0 ? Grp{0, 2, {1, 2}} : Grp{0, 2, {0, 1}};
  const Grp cx1 = px == 0 ? Grp{-1, 1, {0, 0}} : Grp{1, 1, {2, 2}};
  const Grp cx2 = px == 0 ? Grp{0, 2, {1, 2}} : Grp{0, 2, {0, 1}};
  auto mk = [](const Grp& r, const Grp& c, int lo) {
    return UpTap{r.off, c.off, lo, r.n, c.n, {r.idx[0], r.idx[1]}, {c.idx[0], c.idx[1]}};
  };
  // weight stages of 3, 3 and 1 taps
  t[0] = mk(ry1, cx1, 0);
  t[1] = mk(ry1, cx2, 0);
  t[2] = mk(ry1, cx2, 1);
  t[3] = mk(ry2, cx1, 0);
  t[4] = mk(ry2, cx1, 1);
  t[5] = mk(ry2, cx2, 0);
  t[6] = mk(ry2, cx2, 1);
}

std::vector<int> band_rows(int h, int n) {
  std::vector<int> r(n, h / n);
  for (int i = 0; i < h % n; ++i) r[i] += 1;
  return r;
}

int round_up(int a, int b) { return (a + b - 1) / b * b; }

// Placeholder output of dry walks (planning, op descriptions): never dereferenced,
// it only marks the last conv as writing the caller's channels-first output.
char kDryOutTag;
void* const kDryOut = &kDryOutTag;

}  // namespace

struct vaedec {
  vaedec_config cfg{};
  int device = 0;        // the CUDA device current at create: weights, workspace and launches live there
  int dtype = kBF16;
  size_t es = 2;
  std::map<std::string, DevConv> conv;
  std::map<std::string, DevNorm> norm;
  std::vector<void*> allocs;
  // workspace: one arena holding every activation and the attention's scratch (Q, K, V^T, key-split
  // partials, width-band gathers; the fp32 path's scores) as slots whose offsets come from a liveness
  // plan made at create time for max_latent (two slots share bytes only if their lifetimes are disjoint)
  void* arena = nullptr;
  size_t arena_bytes = 0;
  std::vector<size_t> slot_off;     // per slot, in the order a decode walk creates them
  std::vector<size_t> slot_bytes;   // planned (max_latent) size of each slot
  size_t act_peak_bytes = 0;        // largest sum of simultaneously live slots in the plan
  // AutoencoderKLFlux2 latent front-end: patch size (1 = none) and the inverse latent BatchNorm
  // per patched channel, scale = sqrt(var + eps) and shift = mean
  int patch = 1;
  float* bn_scale = nullptr;
  float* bn_shift = nullptr;
  GnPartial* gn_part = nullptr;
  size_t part_elems = 0;
  float* gn_scale = nullptr;
  float* gn_shift = nullptr;
  size_t sc_elems = 0;
  void* io_latent = nullptr;
  void* io_out = nullptr;
  size_t io_latent_bytes = 0, io_out_bytes = 0;
  int* status = nullptr;
  size_t ws_bytes = 0;
  // instrumentation
  unsigned long long launches = 0;
  bool profile = false;
  std::vector<cudaEvent_t> prof_ev;   // 2 per op
  int prof_ops = 0;

  vaedec_status dalloc(void** p, size_t bytes, const char* what) {
    *p = nullptr;
    if (bytes == 0) return VAEDEC_OK;
    if (fault_now(1)) return fail(VAEDEC_ERR_OOM, std::string("injected allocation failure for ") + what);
    cudaError_t e = cudaMalloc(p, bytes);
    if (e != cudaSuccess) {
      cudaGetLastError();
      *p = nullptr;
      return fail(VAEDEC_ERR_OOM, std::string("cudaMalloc failed for ") + what + " (" + std::to_string(bytes) +
                                      " bytes): " + cudaGetErrorString(e));
    }
    allocs.push_back(*p);
    return VAEDEC_OK;
  }
  ~vaedec() {
    for (cudaEvent_t e : prof_ev) cudaEventDestroy(e);
    for (void* p : allocs) cudaFree(p);
  }
};

namespace {

// Sizes a dry walk records for workspace planning.
struct SlotUse {
  size_t bytes;
  long long first, last;   // walk ticks of the slot's creation and of its last use
};
struct Plan {
  size_t part = 0, sc = 0;
  std::vector<SlotUse> slots;
};

// Offsets of the slots in one arena: largest first, each at the lowest 256-byte-aligned offset
// that overlaps no placed slot whose lifetime overlaps its own.  Returns the arena size and the
// largest sum of live slot bytes at any tick (a lower bound on any placement).
size_t place_slots(const std::vector<SlotUse>& slots, std::vector<size_t>* off, size_t* peak_live) {
  const size_t n = slots.size();
  std::vector<size_t> order(n), sz(n);
  for (size_t i = 0; i < n; ++i) {
    order[i] = i;
    sz[i] = (slots[i].bytes + kSlotAlign - 1) / kSlotAlign * kSlotAlign;
  }
  std::stable_sort(order.begin(), order.end(), [&](size_t a, size_t b) {
    if (sz[a] != sz[b]) return sz[a] > sz[b];
    return slots[a].first < slots[b].first;
  });
  off->assign(n, 0);
  std::vector<size_t> placed;
  size_t top = 0;
  for (size_t i : order) {
    std::vector<std::pair<size_t, size_t>> busy;   // [begin, end) of placed slots alive at the same time
    for (size_t j : placed)
      if (!(slots[j].last < slots[i].first || slots[i].last < slots[j].first))
        busy.emplace_back((*off)[j], (*off)[j] + sz[j]);
    std::sort(busy.begin(), busy.end());
    size_t o = 0;
    for (const auto& b : busy) {
      if (o + sz[i] <= b.first) break;
      o = std::max(o, b.second);
    }
    (*off)[i] = o;
    top = std::max(top, o + sz[i]);
    placed.push_back(i);
  }
  // peak of the live bytes over the ticks where some slot begins
  size_t peak = 0;
  for (size_t i = 0; i < n; ++i) {
    size_t live = 0;
    for (size_t j = 0; j < n; ++j)
      if (slots[j].first <= slots[i].first && slots[i].first <= slots[j].last) live += sz[j];
    peak = std::max(peak, live);
  }
  *peak_live = peak;
  return top;
}

class Walker {
 public:
  // axis: 0 = height row bands, 1 = width column bands (on one GPU only attention's query
  // partition depends on it, and no result does)
  Walker(vaedec* h, cudaStream_t st, bool dry, int n_bands, int axis = 0)
      : h_(h), st_(st), dry_(dry), n_bands_(n_bands), axis_(axis), odt_(h->dtype), sdt_(kF32) {}

  // configuration of a debug stop
  int stop_at = -1;
  std::string* desc_out = nullptr;
  void* d_in = nullptr;
  void* d_aux = nullptr;
  void* d_out = nullptr;
  size_t in_b = 0, aux_b = 0, out_b = 0;
  Plan* plan = nullptr;

  vaedec_status status = VAEDEC_OK;
  bool stopped = false;
  int n_ops = 0;

  bool live() const { return status == VAEDEC_OK && !stopped; }

  vaedec_status run(const void* latent, const int64_t* shape, int ndim, void* out) {
    Act z;
    z.B = (int)shape[0];
    z.C = (int)shape[1];
    if (ndim == 5) {
      z.T = (int)shape[2];
      z.H = (int)shape[3];
      z.W = (int)shape[4];
    } else {
      z.T = 1;
      z.H = (int)shape[2];
      z.W = (int)shape[3];
    }
    z.dt = odt_;
    Act x = latent_in(latent, z);
    if (h_->cfg.family == VAEDEC_FAMILY_KL2D)
      walk_kl(x, out);
    else
      walk_wan(x, out);
    return status;
  }

 private:
  vaedec* h_;
  cudaStream_t st_;
  bool dry_;
  int n_bands_;
  int axis_;
  int odt_;   // operand dtype: what the MMAs read (the model dtype)
  int sdt_;   // storage dtype of the residual stream and every pre-norm tensor (fp32)
  int nest_ = 0;
  long long stats_epoch_ = 0;   // bumped whenever a conv rewrites the moments buffer
  int n_slots_ = 0;             // workspace slots created so far by this walk
  long long tick_ = 0;          // walk clock for slot lifetimes (creations and uses)

  bool mixed() const { return odt_ != sdt_; }

  // ---------------------------------------------------------------- helpers
  void* slot_ptr(int slot) const {
    if (dry_ || slot < 0 || slot >= (int)h_->slot_off.size()) return nullptr;
    return static_cast<char*>(h_->arena) + h_->slot_off[slot];
  }
  void* ptr(const Act& a) const { return a.buf >= 0 ? slot_ptr(a.slot) : a.ext; }

  // A new workspace slot of `b` bytes.  The walk creates slots in the same order for every latent
  // shape up to max_latent (no slot depends on the geometry), so the create-time plan gives each
  // one an offset whose bytes no other slot alive at the same time uses.
  int new_slot(size_t b) {
    if (!live()) return -1;   // a stopped walk (debug stop, error) creates nothing more
    const int id = n_slots_++;
    const long long t = ++tick_;
    if (plan) {
      plan->slots.push_back(SlotUse{b, t, t});
    } else if (id >= (int)h_->slot_bytes.size() || b > h_->slot_bytes[id]) {
      set_err(VAEDEC_ERR_INVALID_ARG, "internal: the workspace plan does not cover this decode");
    }
    return id;
  }
  // Marks a slot (or an arena tensor) as read or written now: its bytes stay reserved until then.
  void use_slot(int slot) {
    const long long t = ++tick_;
    if (plan && slot >= 0 && slot < (int)plan->slots.size()) plan->slots[slot].last = t;
  }
  void use(const Act& a) {
    if (a.buf >= 0) use_slot(a.slot);
  }
  static size_t esz(int dt) { return dt == kBF16 ? 2 : 4; }
  size_t bytes(const Act& a) const { return (size_t)a.pixels() * a.C * esz(a.dt); }
  static const char* dts(int dt) { return dt == kBF16 ? "bf16" : "f32"; }

  static int pick(std::initializer_list<int> busy) {
    for (int i = 0; i < kNumAct; ++i)
      if (std::find(busy.begin(), busy.end(), i) == busy.end()) return i;
    return -1;
  }

  // Gives a freshly produced arena tensor its slot (sized for it, alive from now).
  void note_act(Act& a) {
    if (a.buf >= 0) a.slot = new_slot(bytes(a));
  }

  void set_err(vaedec_status s, const std::string& m) {
    if (status == VAEDEC_OK) {
      status = s;
      g_err = m;
    }
  }

  void check(cudaError_t e, const std::string& where) {
    if (e != cudaSuccess && status == VAEDEC_OK) {
      status = VAEDEC_ERR_CUDA;
      g_err = where + ": " + cudaGetErrorString(e);
    }
  }

  static std::string shp(const Act& a) {
    std::ostringstream o;
    o << a.B << "," << a.T << "," << a.H << "," << a.W << "," << a.C;
    return o.str();
  }

  static std::string io(const Act& x, const Act* aux, const Act& y) {
    std::string s = " in=" + shp(x) + " in_dt=" + dts(x.dt) + " out=" + shp(y) + " out_dt=" + dts(y.dt);
    if (aux) s += std::string(" aux=") + shp(*aux) + " aux_dt=" + dts(aux->dt);
    return s;
  }

  // Begin a traced op.  Returns true if its kernels should be enqueued.
  bool begin(const std::string& desc) {
    if (!live()) return false;
    if (nest_ > 0) return !dry_;
    const int idx = n_ops++;
    if (idx == stop_at && desc_out) *desc_out = desc;
    if (!dry_ && h_->profile) {
      while ((int)h_->prof_ev.size() < 2 * (idx + 1)) {
        cudaEvent_t e;
        if (cudaEventCreate(&e) != cudaSuccess) {
          set_err(VAEDEC_ERR_CUDA, "cudaEventCreate failed");
          return false;
        }
        h_->prof_ev.push_back(e);
      }
      check(cudaEventRecord(h_->prof_ev[2 * idx], st_), "profile event");
      h_->prof_ops = idx + 1;
    }
    return !dry_;
  }

  void count(int n = 1) {
    if (dry_) return;
    for (int i = 0; i < n; ++i)
      if (fault_now(2)) set_err(VAEDEC_ERR_CUDA, "injected launch failure");
    h_->launches += (unsigned long long)n;
  }

  // End a traced op: at the stop op, copy its activations out and stop.
  void end(const Act* in, const Act* aux, const Act& out_act) {
    if (nest_ > 0 || !live()) return;
    const int idx = n_ops - 1;
    if (!dry_ && h_->profile && 2 * idx + 1 < (int)h_->prof_ev.size())
      check(cudaEventRecord(h_->prof_ev[2 * idx + 1], st_), "profile event");
    if (idx != stop_at) return;
    if (!dry_) {
      auto cp = [&](void* dst, size_t cap, const Act* a, const char* what) {
        if (dst == nullptr || a == nullptr) return;
        const size_t n = bytes(*a);
        if (cap < n) {
          set_err(VAEDEC_ERR_INVALID_ARG, std::string("debug buffer too small for ") + what);
          return;
        }
        check(cudaMemcpyAsync(dst, ptr(*a), n, cudaMemcpyDeviceToDevice, st_), "debug copy");
      };
      cp(d_in, in_b, in, "input");
      cp(d_aux, aux_b, aux, "aux");
      cp(d_out, out_b, &out_act, "output");
    }
    stopped = true;
  }

  const DevConv* W(const std::string& name) {
    auto it = h_->conv.find(name);
    if (it == h_->conv.end()) {
      set_err(VAEDEC_ERR_INVALID_ARG, "missing weights for " + name);
      return nullptr;
    }
    return &it->second;
  }
  const DevNorm* N(const std::string& name) {
    auto it = h_->norm.find(name);
    if (it == h_->norm.end()) {
      set_err(VAEDEC_ERR_INVALID_ARG, "missing norm parameters for " + name);
      return nullptr;
    }
    return &it->second;
  }

  // ---------------------------------------------------------------- ops
  Act latent_in(const void* latent, const Act& z) {
    const int p = h_->patch;
    Act y = z;
    y.buf = 0;
    y.dt = odt_;
    y.C = z.C / (p * p);   // the front-end's unpatchify (p = 1: a plain layout change)
    y.H = z.H * p;
    y.W = z.W * p;
    note_act(y);
    Act zin = z;
    zin.buf = -1;
    zin.ext = const_cast<void*>(latent);
    if (begin("kind=latent name=latent" + io(zin, nullptr, y))) {
      count();
      if (p > 1)
        check(launch_latent_frontend(odt_, latent, ptr(y), z.B, y.C, z.H, z.W, p, h_->bn_scale, h_->bn_shift, st_),
              "latent front-end");
      else
        check(launch_to_channels_last(odt_, latent, ptr(y), z.B, z.C, (long long)z.T * z.H * z.W, st_),
              "latent layout");
    }
    end(&zin, nullptr, y);
    return y;
  }

  // A 1x1 convolution that runs as the channel-major GEMM (bf16 path).
  bool gemm_conv(const ConvGeom& g, bool rowscale, bool residual, bool out2) const {
    return h_->dtype == kBF16 && g.ntaps == 1 && g.nphase == 1 && g.time_up_c == 0 && g.osx == 1 && g.osy == 1 &&
           !rowscale && g.gn_part == nullptr && g.oT == g.T && g.oH == g.H && g.oW == g.W &&
           (!g.out_chfirst || (!residual && !out2));
  }

  // Name of the kernel `launch` will run for a conv op (recorded in the op description).
  const char* conv_kernel(const ConvGeom& g, bool residual, bool out2, bool narrow_w) const {
    if (h_->dtype != kBF16) return "conv_simple_f32";
    if (gemm_conv(g, false, residual, out2)) return "gemm_cm";
    if (narrow_w && !residual && !out2 && g.gn_part == nullptr && conv_narrow_applicable(g)) return "conv_narrow";
    if (conv_halo_t_applicable(g)) return "conv_halo_t";
    if (conv_halo_applicable(g)) return "conv_halo";
    return "conv_tc";
  }

  // Launch one GEMM/conv described by `g`.
  int launch(const ConvGeom& g, const void* in, const DevConv& w, const void* wptr, const float* bias,
             const void* residual, const float* rowscale, void* out, void* out2, const char* what,
             const ConvShortcut* sc = nullptr) {
    count();
    if (g.gn_part != nullptr) ++stats_epoch_;   // the moments buffer is about to be rewritten
    int gn_chunks = 0;
    if (sc == nullptr && gemm_conv(g, rowscale != nullptr, residual != nullptr, out2 != nullptr)) {
      // 1x1 convolution = channel-major GEMM: out[pixel][co] = W[co][:] . in[pixel][:]
      const long long S = (long long)g.H * g.W;
      GemmArgs a;
      a.K = g.Cin;
      a.out_f32 = g.out_f32;
      a.scale = g.scale;
      a.residual = residual;
      a.res_f32 = g.res_f32;
      a.out2 = out2;
      if (!g.out_chfirst) {
        a.A = wptr;
        a.lda = (long long)w.ntaps * g.Cin;
        a.M = g.Cout;
        a.B = in;
        a.ldb = g.Cin;
        a.N = (int)((long long)g.B * g.T * S);
        a.out = out;
        a.ldo = g.oC;
        a.bias_m = bias;
        gemm(a, what, false);
      } else {
        // channels-first output: per frame, pixels on M and channels on N
        const size_t ies = esz(h_->dtype), oes = g.out_f32 ? 4 : 2;
        for (long long f = 0; f < (long long)g.B * g.T && live(); ++f) {
          GemmArgs af = a;
          af.A = static_cast<const char*>(in) + (size_t)(f * S * g.Cin) * ies;
          af.lda = g.Cin;
          af.M = (int)S;
          af.B = wptr;
          af.ldb = (long long)w.ntaps * g.Cin;
          af.N = g.Cout;
          af.out = static_cast<char*>(out) + (size_t)(f * g.oC * S) * oes;
          af.ldo = S;
          af.bias_n = bias;
          gemm(af, what, f > 0);
        }
      }
      return 0;
    }
    if (sc == nullptr && h_->dtype == kBF16 && w.wn != nullptr && wptr == w.w && residual == nullptr &&
        rowscale == nullptr && out2 == nullptr && g.gn_part == nullptr && conv_narrow_applicable(g)) {
      const char* why = nullptr;
      cudaError_t e = launch_conv_narrow(g, in, w.wn, bias, out, h_->status, st_, &why);
      if (e != cudaSuccess) set_err(VAEDEC_ERR_CUDA, std::string(what) + ": " + (why ? why : cudaGetErrorString(e)));
      return 0;
    }
    if (h_->dtype == kBF16) {
      const char* why = nullptr;
      cudaError_t e = launch_conv_tc(g, in, wptr, w.ntaps, w.rows, bias, residual, rowscale, out, out2, h_->status,
                                     st_, &why, &gn_chunks, sc);
      if (e != cudaSuccess) set_err(VAEDEC_ERR_CUDA, std::string(what) + ": " + (why ? why : cudaGetErrorString(e)));
    } else {
      check(launch_conv_simple_f32(g, static_cast<const float*>(in), static_cast<const float*>(wptr), w.ntaps, bias,
                                   static_cast<const float*>(residual), rowscale, static_cast<float*>(out), st_),
            what);
    }
    return gn_chunks;
  }

  // Launch one channel-major tensor-core GEMM (bf16 path only).
  void gemm(const GemmArgs& a, const char* what, bool count_it = true) {
    if (count_it) count();
    const char* why = nullptr;
    cudaError_t e = launch_gemm_cm(a, h_->status, st_, &why);
    if (e != cudaSuccess) set_err(VAEDEC_ERR_CUDA, std::string(what) + ": " + (why ? why : cudaGetErrorString(e)));
  }

  // The exact two-by-two phase form of an upsample conv (weights w.wup).
  static void fill_taps_up7(ConvGeom& g) {
    std::memset(g.taps, 0, sizeof(g.taps));
    g.nphase = 4;
    g.ntaps = kUpTaps;
    for (int ph = 0; ph < 4; ++ph) {
      UpTap t[kUpTaps];
      up_phase_taps(ph, t);
      for (int k = 0; k < kUpTaps; ++k)
        g.taps[ph][k] = ConvTap{0, (int8_t)t[k].oy, (int8_t)t[k].ox, (int8_t)(ph * kUpTaps + k)};
    }
  }

  static void fill_taps(ConvGeom& g, ConvKind kind, const DevConv& w) {
    std::memset(g.taps, 0, sizeof(g.taps));
    g.nphase = 1;
    if (kind == K1) {
      g.ntaps = 1;
      g.taps[0][0] = ConvTap{0, 0, 0, 0};
    } else if (kind == K3) {
      g.ntaps = 9;
      for (int i = 0; i < 3; ++i)
        for (int j = 0; j < 3; ++j)
          g.taps[0][i * 3 + j] = ConvTap{0, (int8_t)(i - 1), (int8_t)(j - 1), (int8_t)(i * 3 + j)};
    } else if (kind == C3) {
      g.ntaps = w.kt * w.kh * w.kw;
      for (int s = 0; s < w.kt; ++s)
        for (int i = 0; i < w.kh; ++i)
          for (int j = 0; j < w.kw; ++j) {
            const int k = (s * w.kh + i) * w.kw + j;
            g.taps[0][k] = ConvTap{(int8_t)(s - (w.kt - 1)), (int8_t)(i - w.kh / 2), (int8_t)(j - w.kw / 2), (int8_t)k};
          }
    } else if (kind == TIME) {
      g.ntaps = w.kt;
      for (int s = 0; s < w.kt; ++s) g.taps[0][s] = ConvTap{(int8_t)(s - (w.kt - 1)), 0, 0, (int8_t)s};
    } else {  // UP: nearest-2x then 3x3, as four phases on the low-resolution grid
      g.nphase = 4;
      g.ntaps = 9;
      for (int ph = 0; ph < 4; ++ph) {
        const int py = ph >> 1, px = ph & 1;
        for (int i = 0; i < 3; ++i)
          for (int j = 0; j < 3; ++j) {
            const int oy = (py + i - 1) >= 0 ? (py + i - 1) / 2 : -1;   // floor((py + i - 1) / 2)
            const int ox = (px + j - 1) >= 0 ? (px + j - 1) / 2 : -1;
            g.taps[ph][i * 3 + j] = ConvTap{0, (int8_t)oy, (int8_t)ox, (int8_t)(i * 3 + j)};
          }
      }
    }
  }

  // conv op: x (operand dtype) -> y (`out_dt`, channels-last buffer `out_buf`, or the
  // final channels-first output).  `copy` (optional) receives a bf16 copy of y.
  Act conv(const Act& x, const std::string& name, ConvKind kind, const Act* res, int out_buf, int out_dt,
           void* final_out = nullptr, Act* copy = nullptr, int copy_buf = -1, bool want_stats = false,
           const Act* sc_x = nullptr, const std::string& sc_name = std::string()) {
    Act y = x;
    y.stats_chunks = 0;
    y.stats_epoch = -1;
    const DevConv* w = W(name);
    if (!w || !live()) return y;
    if (w->cin != x.C) {
      set_err(VAEDEC_ERR_INVALID_ARG, "channel mismatch at " + name);
      return y;
    }
    if (x.dt != odt_) {
      set_err(VAEDEC_ERR_INVALID_ARG, "internal: conv operand in the wrong dtype at " + name);
      return y;
    }
    y.buf = final_out ? -1 : out_buf;
    y.ext = final_out;
    y.dt = final_out ? odt_ : out_dt;
    y.C = (kind == TIME) ? w->cout / 2 : w->cout;
    if (kind == UP) {
      y.H *= 2;
      y.W *= 2;
    }
    if (kind == TIME) y.T = 2 * x.T - 1;
    note_act(y);
    Act yc;
    if (copy) {
      yc = y;
      yc.buf = copy_buf;
      yc.dt = kBF16;
      note_act(yc);
      *copy = yc;
    }
    // inputs are read after the outputs exist, and the outputs stay reserved to the end of the op:
    // no two tensors of one op share bytes
    use(x);
    if (res) use(*res);
    if (sc_x) use(*sc_x);
    use(y);
    if (copy) use(yc);
    ConvGeom g;
    std::memset(&g, 0, sizeof(g));
    {
      g.B = x.B;
      g.T = x.T;
      g.H = x.H;
      g.W = x.W;
      g.Cin = x.C;
      g.Cout = w->cout;
      fill_taps(g, kind, *w);
      g.oT = y.T;
      g.oH = y.H;
      g.oW = y.W;
      g.oC = y.C;
      g.osy = g.osx = (kind == UP) ? 2 : 1;
      g.time_up_c = (kind == TIME) ? y.C : 0;
      g.out_chfirst = final_out ? 1 : 0;
      g.out_f32 = y.dt == kF32 ? 1 : 0;
      g.res_f32 = (res && res->dt == kF32) ? 1 : 0;
      g.scale = 1.f;
    }
    // an upsample conv runs in its exact two-by-two phase form where the channel-major kernel takes
    // it (7 weight taps per phase instead of 9)
    DevConv wrun = *w;
    bool up7 = false;
    if (kind == UP && w->wup != nullptr) {
      ConvGeom g7 = g;
      fill_taps_up7(g7);
      if (conv_halo_t_applicable(g7)) {
        g = g7;
        wrun.w = w->wup;
        wrun.ntaps = 4 * kUpTaps;
        up7 = true;
      }
    }
    // a fused 1x1 shortcut (sc_x, weights sc_name) adds its flops and uses the combined bias
    const DevConv* scw = sc_x ? W(sc_name) : nullptr;
    if (sc_x && (!scw || !w->b_sc)) return y;
    double flops = conv_flops(x, y, *w, kind);
    if (scw) flops += 2.0 * (double)y.pixels() * scw->cout * scw->cin;
    // multiply-adds the tensor cores execute (the exact phase form: 7 of the 9 taps' worth)
    const double exec_flops = up7 ? flops * kUpTaps / 9.0 : flops;
    std::ostringstream d;
    d << "kind=conv name=" << name << " conv="
      << (kind == K3 ? "k3" : kind == K1 ? "k1" : kind == C3 ? "causal3" : kind == UP ? "up2x_k3" : "time")
      << io(x, sc_x ? sc_x : res, y) << " res=" << (res ? 1 : 0) << " final=" << (final_out ? 1 : 0)
      << " taps=" << w->ntaps << " flops=" << flops << " exec_flops=" << exec_flops
      << " kernel=" << (scw ? "conv_halo_t" : conv_kernel(g, res != nullptr, copy != nullptr, w->wn != nullptr));
    if (scw) d << " shortcut=" << sc_name;
    if (begin(d.str())) {
      const char* in = static_cast<const char*>(ptr(x));
      void* out2 = copy ? ptr(yc) : nullptr;
      if (kind == TIME) {
        // frame 0 passes through; frames 1..T-1 feed the causal time conv
        if (y.dt != x.dt) set_err(VAEDEC_ERR_INVALID_ARG, "internal: time upsample dtype");
        const size_t frame = (size_t)x.H * x.W * x.C * esz(x.dt);
        check(cudaMemcpy2DAsync(ptr(y), frame * y.T, in, frame * x.T, frame, x.B, cudaMemcpyDeviceToDevice, st_),
              "frame 0 copy");
        // the time-conv view starts at frame 1 with T-1 frames while the sample
        // stride stays T frames: one launch per sample
        for (int b = 0; b < x.B && x.T > 1 && live(); ++b) {
          ConvGeom gb = g;
          gb.B = 1;
          gb.T = x.T - 1;
          const size_t in_off = (size_t)b * x.T * frame + frame;
          const size_t out_off = (size_t)b * y.T * y.H * y.W * y.C * esz(y.dt);
          launch(gb, in + in_off, *w, w->w, w->b, nullptr, nullptr, static_cast<char*>(ptr(y)) + out_off, nullptr,
                 name.c_str());
        }
      } else {
        // moments for a following GroupNorm, when the kernel can write them in its epilogue
        if (want_stats && h_->cfg.family == VAEDEC_FAMILY_KL2D && h_->dtype == kBF16 && y.dt == kF32) {
          g.gn_part = h_->gn_part;
          g.gn_groups = h_->cfg.norm_groups;
        }
        ConvShortcut csc;
        if (scw) {
          csc.in = ptr(*sc_x);
          csc.w = scw->w;
          csc.cin = scw->cin;
          csc.w_rows = scw->rows;
        }
        const int chunks = launch(g, in, wrun, wrun.w, scw ? w->b_sc : w->b, res ? ptr(*res) : nullptr, nullptr,
                                  ptr(y), out2, name.c_str(), scw ? &csc : nullptr);
        if (chunks > 0) {
          y.stats_chunks = chunks;
          y.stats_epoch = ++stats_epoch_;
        }
      }
    }
    end(&x, sc_x ? sc_x : res, y);
    return y;
  }

  // Algorithmic multiply-add work of a conv op (2 flops per MAC): every output
  // element is a dot product over taps x C_in (the upsampled conv counts its
  // 3x3 taps on the high-resolution output, the time conv its frames 1..T-1).
  static double conv_flops(const Act& x, const Act& y, const DevConv& w, ConvKind kind) {
    double out_pix = (double)y.pixels();
    double n = (double)w.cout;
    if (kind == TIME) {
      out_pix = (double)x.B * (x.T - 1) * x.H * x.W;   // time-conv outputs (2C channels each)
    }
    return 2.0 * out_pix * n * (double)w.ntaps * (double)x.C;
  }

  // GroupNorm: x (any dtype) -> operand dtype; `raw` (optional) receives x cast.
  Act group_norm(const Act& x, const std::string& prefix, bool silu, int out_buf, Act* raw = nullptr,
                 int raw_buf = -1) {
    Act y = x;
    y.buf = out_buf;
    y.dt = odt_;
    y.stats_chunks = 0;
    y.stats_epoch = -1;
    const DevNorm* n = N(prefix);
    if (!n || !live()) return y;
    const int G = h_->cfg.norm_groups;
    const int rows = x.T * x.H;
    // moments from the producing conv's epilogue, if they are still the newest ones
    const bool have = x.stats_chunks > 0 && x.stats_epoch == stats_epoch_;
    const int n_chunks = have ? x.stats_chunks : rows;
    if (plan) {
      // fused chunks: at most 2 phase columns x ceil(W / 96) + 1 pixel tiles per output row
      plan->part = std::max(plan->part, (size_t)x.B * rows * (size_t)(2 * (x.W / 96 + 2)) * G);
      plan->sc = std::max(plan->sc, (size_t)x.B * x.C);
    }
    note_act(y);
    Act yr;
    if (raw) {
      yr = x;
      yr.buf = raw_buf;
      yr.dt = odt_;
      note_act(yr);
      *raw = yr;
    }
    use(x);
    use(y);
    if (raw) use(yr);
    if (begin("kind=groupnorm name=" + prefix + io(x, nullptr, y) + " silu=" + (silu ? "1" : "0") +
              " groups=" + std::to_string(G) + " fused_stats=" + (have ? "1" : "0"))) {
      count(have ? 2 : 3);
      if (!have) {
        check(launch_gn_partials(x.dt, ptr(x), x.B, rows, x.W, x.C, G, 1, h_->gn_part, st_), "gn partials");
        ++stats_epoch_;
      }
      check(launch_gn_finalize(h_->gn_part, x.B, n_chunks, x.C, G, n->g, n->b, h_->cfg.eps, h_->gn_scale,
                               h_->gn_shift, st_),
            "gn finalize");
      check(launch_gn_apply(x.dt, y.dt, ptr(x), ptr(y), raw ? ptr(yr) : nullptr, (long long)x.T * x.H * x.W, x.B,
                            x.C, h_->gn_scale, h_->gn_shift, silu ? 1 : 0, st_),
            "gn apply");
    }
    end(&x, nullptr, y);
    return y;
  }

  Act rms_norm(const Act& x, const std::string& prefix, bool silu, int out_buf, Act* raw = nullptr,
               int raw_buf = -1) {
    Act y = x;
    y.stats_chunks = 0;
    y.stats_epoch = -1;
    y.buf = out_buf;
    y.dt = odt_;
    const DevNorm* n = N(prefix);
    if (!n || !live()) return y;
    note_act(y);
    Act yr;
    if (raw) {
      yr = x;
      yr.buf = raw_buf;
      yr.dt = odt_;
      note_act(yr);
      *raw = yr;
    }
    use(x);
    use(y);
    if (raw) use(yr);
    if (begin("kind=rmsnorm name=" + prefix + io(x, nullptr, y) + " silu=" + (silu ? "1" : "0"))) {
      count();
      check(launch_rms_norm(x.dt, y.dt, ptr(x), ptr(y), raw ? ptr(yr) : nullptr, x.pixels(), x.C, n->g,
                            silu ? 1 : 0, st_),
            "rms norm");
    }
    end(&x, nullptr, y);
    return y;
  }

  // Attention block over frames (B*T sequences of H*W tokens) with band-local queries.
  Act attention(const Act& x, const std::string& prefix, bool wan) {
    const int a_buf = pick({x.buf});
    const int o_buf = pick({x.buf, a_buf});
    Act y = x;
    y.buf = o_buf;
    y.dt = sdt_;
    y.stats_chunks = 0;
    y.stats_epoch = -1;
    const int C = x.C;
    const long long Ntok = (long long)x.H * x.W;
    const int F = x.B * x.T;   // sequences
    const size_t oes = esz(odt_);
    note_act(y);
    // the op's scratch, alive for this op only: Q, K, V^T, the width bands' gathered queries and
    // their output before the scatter, and the bf16 path's key-split partials or the fp32 path's
    // scores, probabilities and row sums of its largest band (the plan walks one band)
    const size_t qkv_b = (size_t)F * (size_t)Ntok * (size_t)C * oes;
    const int s_q = new_slot(qkv_b), s_k = new_slot(qkv_b), s_vt = new_slot(qkv_b);
    const int s_qg = new_slot(qkv_b), s_ob = new_slot(qkv_b);
    int s_work = -1, s_s = -1, s_p = -1, s_l = -1;
    if (h_->dtype == kBF16) {
      s_work = new_slot(flash_work_bytes(F, Ntok, C));
    } else {
      int maxp = 0;
      for (int r : band_rows(axis_ == 1 ? x.W : x.H, n_bands_)) maxp = std::max(maxp, r);
      const size_t nrmax = (size_t)maxp * (size_t)(axis_ == 1 ? x.H : x.W);
      s_s = new_slot(nrmax * (size_t)Ntok * sizeof(float));
      s_p = new_slot(nrmax * (size_t)Ntok * oes);
      s_l = new_slot(nrmax * sizeof(float));
    }
    void* const attn_q = slot_ptr(s_q);
    void* const attn_k = slot_ptr(s_k);
    void* const attn_vt = slot_ptr(s_vt);
    void* const attn_qg = slot_ptr(s_qg);
    void* const attn_ob = slot_ptr(s_ob);
    void* const attn_work = slot_ptr(s_work);
    float* const attn_s = static_cast<float*>(slot_ptr(s_s));
    void* const attn_p = slot_ptr(s_p);
    float* const attn_l = static_cast<float*>(slot_ptr(s_l));
    // projections 4 x (2 N C^2) plus scores and probabilities x values 2 x (2 N^2 C), per sequence
    const double attn_flops = (double)F * (8.0 * (double)Ntok * C * C + 4.0 * (double)Ntok * (double)Ntok * C);
    std::ostringstream fl;
    fl << attn_flops;
    const bool run = begin("kind=attention name=" + prefix + io(x, nullptr, y) + " wan=" + (wan ? "1" : "0") +
                           " bands=" + std::to_string(n_bands_) + " flops=" + fl.str());
    ++nest_;
    if (live()) {
      // normalisation (GroupNorm for KL, channel RMSNorm for Wan), no SiLU
      Act hn = wan ? rms_norm(x, prefix + ".norm", false, a_buf) : group_norm(x, prefix + ".group_norm", false, a_buf);
      DevConv wq, wk, wv, wo;
      bool ok = true;
      if (wan) {
        const DevConv* qkv = W(prefix + ".to_qkv");
        const DevConv* pr = W(prefix + ".proj");
        ok = qkv && pr;
        if (ok) {
          const size_t blk = (size_t)C * qkv->ntaps * qkv->cin * oes;
          wq = wk = wv = *qkv;
          wq.cout = wk.cout = wv.cout = C;
          wq.rows = wk.rows = wv.rows = C;
          wk.w = static_cast<char*>(qkv->w) + blk;
          wv.w = static_cast<char*>(qkv->w) + 2 * blk;
          wk.b = qkv->b + C;
          wv.b = qkv->b + 2 * C;
          wo = *pr;
        }
      } else {
        const DevConv *a = W(prefix + ".to_q"), *b = W(prefix + ".to_k"), *c = W(prefix + ".to_v"),
                      *d = W(prefix + ".to_out.0");
        ok = a && b && c && d;
        if (ok) {
          wq = *a;
          wk = *b;
          wv = *c;
          wo = *d;
        }
      }
      if (ok && run) {
        // projections on a (F, 1, H, W) grid: Q, K channels-last, V channels-first (V^T per frame)
        ConvGeom g;
        std::memset(&g, 0, sizeof(g));
        g.B = F;
        g.T = 1;
        g.H = x.H;
        g.W = x.W;
        g.Cin = C;
        g.Cout = C;
        g.nphase = 1;
        g.ntaps = 1;
        g.oT = 1;
        g.oH = x.H;
        g.oW = x.W;
        g.oC = C;
        g.osy = g.osx = 1;
        g.out_f32 = odt_ == kF32;
        g.scale = 1.f;
        launch(g, ptr(hn), wq, wq.w, wq.b, nullptr, nullptr, attn_q, nullptr, "attention q");
        launch(g, ptr(hn), wk, wk.w, wk.b, nullptr, nullptr, attn_k, nullptr, "attention k");
        ConvGeom gv = g;
        gv.out_chfirst = 1;
        launch(gv, ptr(hn), wv, wv.w, wv.b, nullptr, nullptr, attn_vt, nullptr, "attention v");
        // band-local queries against every key/value of the frame; width bands are gathered into a
        // dense query buffer and their output scattered back (each query's arithmetic is the same
        // whichever band holds it)
        const bool wband = axis_ == 1;
        const std::vector<int> rows = band_rows(wband ? x.W : x.H, n_bands_);
        if (h_->dtype == kBF16) {
          // fused tensor-core attention: one launch covers every band of every frame (query tiles
          // never cross a band), then the merge of its key splits
          void* q_src = attn_q;
          void* o_dst = ptr(hn);
          if (wband) {
            // frame f's width band b goes to rows f * Ntok + H * c0 of the gathered buffer
            for (int f = 0; f < F && live(); ++f) {
              int c0 = 0;
              for (int band = 0; band < n_bands_ && live(); ++band) {
                count();
                if (live())
                  check(launch_band_cols(odt_, static_cast<char*>(attn_q) + (size_t)f * Ntok * C * oes,
                                         static_cast<char*>(attn_qg) + ((size_t)f * Ntok + (size_t)x.H * c0) * C * oes,
                                         x.H, x.W, C, c0, rows[band], 1, st_),
                        "attention band gather");
                c0 += rows[band];
              }
            }
            q_src = attn_qg;
            o_dst = attn_ob;
          }
          FlashArgs fa;
          fa.q = q_src;
          fa.k = attn_k;
          fa.vt = attn_vt;
          fa.out = o_dst;
          fa.part = static_cast<float*>(attn_work);
          fa.ml = static_cast<char*>(attn_work) +
                  (size_t)flash_splits(Ntok) * (size_t)F * (size_t)Ntok * (size_t)C * sizeof(float);
          fa.F = F;
          fa.ntok = Ntok;
          fa.C = C;
          fa.U = wband ? x.H : x.W;
          fa.n_seg = n_bands_;
          fa.seg_q = (wband ? x.W : x.H) / n_bands_;
          fa.seg_rem = (wband ? x.W : x.H) % n_bands_;
          if (live()) {
            count();
            const char* why = nullptr;
            cudaError_t e = live() ? launch_attn_flash(fa, h_->status, st_, &why) : cudaSuccess;
            if (e != cudaSuccess)
              set_err(VAEDEC_ERR_CUDA, std::string("attention: ") + (why ? why : cudaGetErrorString(e)));
          }
          if (live() && flash_splits(Ntok) > 1) {
            count();
            if (live()) check(launch_attn_combine(fa, st_), "attention key-split merge");
          }
          if (wband) {
            for (int f = 0; f < F && live(); ++f) {
              int c0 = 0;
              for (int band = 0; band < n_bands_ && live(); ++band) {
                count();
                if (live())
                  check(launch_band_cols(odt_, static_cast<char*>(attn_ob) + ((size_t)f * Ntok + (size_t)x.H * c0) * C * oes,
                                         static_cast<char*>(ptr(hn)) + (size_t)f * Ntok * C * oes, x.H, x.W, C, c0,
                                         rows[band], 0, st_),
                        "attention band scatter");
                c0 += rows[band];
              }
            }
          }
        } else {
          // fp32 path on the CUDA cores: per band, scores = Q K^T / sqrt(C), row softmax, P V
          DevConv kview;
          kview.ntaps = 1;
          kview.cin = C;
          kview.rows = (int)Ntok;
          kview.cout = (int)Ntok;
          DevConv vview;
          vview.ntaps = 1;
          vview.cin = (int)Ntok;
          vview.rows = C;
          vview.cout = C;
          const float scale = 1.f / std::sqrt((float)C);
          for (int f = 0; f < F && live(); ++f) {
            int r0 = 0;
            for (int band = 0; band < n_bands_ && live(); ++band) {
              const int nr = wband ? x.H * rows[band] : rows[band] * x.W;
              // height band: its queries and its output are contiguous rows of the frame (O overwrites
              // the band's normalised rows); width band: gathered / scattered through dense buffers
              const size_t qoff = wband ? 0 : ((size_t)f * Ntok + (size_t)r0 * x.W) * C;
              void* q_band = static_cast<char*>(wband ? attn_qg : attn_q) + qoff * oes;
              void* o_band = wband ? attn_ob : static_cast<void*>(static_cast<char*>(ptr(hn)) + qoff * oes);
              if (wband) {
                count();
                check(launch_band_cols(odt_, static_cast<char*>(attn_q) + (size_t)f * Ntok * C * oes, attn_qg,
                                       x.H, x.W, C, r0, rows[band], 1, st_),
                      "attention band gather");
              }
              ConvGeom gs;
              std::memset(&gs, 0, sizeof(gs));
              gs.B = 1;
              gs.T = 1;
              gs.H = 1;
              gs.W = nr;
              gs.Cin = C;
              gs.Cout = (int)Ntok;
              gs.nphase = 1;
              gs.ntaps = 1;
              gs.oT = 1;
              gs.oH = 1;
              gs.oW = nr;
              gs.oC = (int)Ntok;
              gs.osy = gs.osx = 1;
              gs.out_f32 = 1;
              gs.scale = scale;
              launch(gs, q_band, kview,
                     static_cast<char*>(attn_k) + (size_t)f * Ntok * C * oes, nullptr, nullptr, nullptr,
                     attn_s, nullptr, "attention scores");
              count();
              check(launch_softmax_rows(odt_, attn_s, attn_p, attn_l, nr, (int)Ntok, st_), "softmax");
              ConvGeom go = gs;
              go.Cin = (int)Ntok;
              go.Cout = C;
              go.oC = C;
              go.out_f32 = odt_ == kF32;
              go.scale = 1.f;
              launch(go, attn_p, vview, static_cast<char*>(attn_vt) + (size_t)f * C * Ntok * oes, nullptr,
                     nullptr, attn_l, o_band, nullptr, "attention pv");
              if (wband && live()) {
                count();
                check(launch_band_cols(odt_, o_band, static_cast<char*>(ptr(hn)) + (size_t)f * Ntok * C * oes, x.H,
                                       x.W, C, r0, rows[band], 0, st_),
                      "attention band scatter");
              }
              r0 += rows[band];
            }
          }
        }
        // output projection + residual in fp32
        ConvGeom gp = g;
        gp.out_f32 = y.dt == kF32;
        gp.res_f32 = x.dt == kF32;
        launch(gp, ptr(hn), wo, wo.w, wo.b, ptr(x), nullptr, ptr(y), nullptr, "attention out");
      }
      use(hn);
    }
    use(x);
    use(y);
    for (int sl : {s_q, s_k, s_vt, s_qg, s_ob, s_work, s_s, s_p, s_l})
      if (sl >= 0) use_slot(sl);
    --nest_;
    end(&x, nullptr, y);
    return y;
  }

  // ---------------------------------------------------------------- blocks
  // Residual block on the fp32 stream x.  When `copy` is given, the block output
  // is also stored as a bf16 operand copy (for a following upsample conv).
  // Whether block `p`'s 1x1 shortcut can be fused into its conv2 (bf16 2D path, channel-major
  // halo kernel geometry).
  bool fuse_shortcut(const Act& t2, const std::string& p) const {
    if (h_->dtype != kBF16 || h_->cfg.family != VAEDEC_FAMILY_KL2D) return false;
    auto c2 = h_->conv.find(p + ".conv2");
    auto sc = h_->conv.find(p + ".conv_shortcut");
    if (c2 == h_->conv.end() || sc == h_->conv.end() || c2->second.b_sc == nullptr) return false;
    if (sc->second.ntaps != 1) return false;
    ConvGeom g;
    std::memset(&g, 0, sizeof(g));
    g.B = t2.B;
    g.T = t2.T;
    g.H = t2.H;
    g.W = t2.W;
    g.Cin = t2.C;
    g.Cout = c2->second.cout;
    fill_taps(g, K3, c2->second);
    g.oT = t2.T;
    g.oH = t2.H;
    g.oW = t2.W;
    g.oC = g.Cout;
    g.osy = g.osx = 1;
    return conv_halo_t_applicable(g) && conv_halo_t_shortcut_ok(g, sc->second.cin);
  }

  Act resnet(const Act& x, const std::string& p, bool wan, Act* copy) {
    const bool sc = h_->conv.count(p + ".conv_shortcut") > 0;
    const int tb = pick({x.buf});
    Act xb = x;   // operand copy of x for the shortcut conv
    const bool need_raw = sc && mixed();
    const int rb = need_raw ? pick({x.buf, tb}) : -1;
    Act t = wan ? rms_norm(x, p + ".norm1", true, tb, need_raw ? &xb : nullptr, rb)
                : group_norm(x, p + ".norm1", true, tb, need_raw ? &xb : nullptr, rb);
    const int hb = pick({x.buf, tb, rb});
    Act hh = conv(t, p + ".conv1", wan ? C3 : K3, nullptr, hb, sdt_, nullptr, nullptr, -1, !wan);
    Act t2 = wan ? rms_norm(hh, p + ".norm2", true, tb) : group_norm(hh, p + ".norm2", true, tb);
    if (sc && need_raw && fuse_shortcut(t2, p)) {
      // the 1x1 shortcut runs inside conv2 (extra K over the raw operand copy of x).  Whether it can
      // depends on the geometry, so the workspace slot the separate shortcut output would take is
      // still created (and left unused): the walk's slot sequence stays the same for every shape.
      {
        Act unused = t2;
        unused.buf = 0;
        unused.dt = sdt_;
        unused.C = h_->conv.at(p + ".conv_shortcut").cout;
        note_act(unused);
      }
      if (copy && mixed())
        return conv(t2, p + ".conv2", K3, nullptr, hb, sdt_, nullptr, copy, pick({tb, hb, rb}), true, &xb,
                    p + ".conv_shortcut");
      Act y = conv(t2, p + ".conv2", K3, nullptr, hb, sdt_, nullptr, nullptr, -1, true, &xb, p + ".conv_shortcut");
      if (copy) *copy = y;
      return y;
    }
    Act res = x;
    int scb = -1;
    if (sc) {
      scb = pick({x.buf, tb, hb, rb});
      res = conv(xb, p + ".conv_shortcut", wan ? C3 : K1, nullptr, scb, sdt_);
    }
    const int out_buf = hb;
    if (copy && mixed()) {
      const int cb = sc ? pick({tb, hb, scb}) : pick({x.buf, tb, hb});
      return conv(t2, p + ".conv2", wan ? C3 : K3, &res, out_buf, sdt_, nullptr, copy, cb, !wan);
    }
    Act y = conv(t2, p + ".conv2", wan ? C3 : K3, &res, out_buf, sdt_, nullptr, nullptr, -1, !wan);
    if (copy) *copy = y;
    return y;
  }

  void walk_kl(Act x, void* out) {
    const vaedec_config& c = h_->cfg;
    x = conv(x, "conv_in", K3, nullptr, pick({x.buf}), sdt_, nullptr, nullptr, -1, true);
    x = resnet(x, "mid_block.resnets.0", false, nullptr);
    x = attention(x, "mid_block.attentions.0", false);
    x = resnet(x, "mid_block.resnets.1", false, nullptr);
    for (int s = 0; s < c.n_stages && live(); ++s) {
      const std::string pre = "up_blocks." + std::to_string(s);
      Act xc;
      for (int r = 0; r < c.stage_resnets[s]; ++r) {
        const bool last = (r + 1 == c.stage_resnets[s]) && c.stage_upsample[s];
        x = resnet(x, pre + ".resnets." + std::to_string(r), false, last ? &xc : nullptr);
      }
      if (c.stage_upsample[s])
        x = conv(xc, pre + ".upsamplers.0.conv", UP, nullptr, pick({x.buf, xc.buf}), sdt_, nullptr, nullptr, -1, true);
    }
    Act t = group_norm(x, "conv_norm_out", true, pick({x.buf}));
    conv(t, "conv_out", K3, nullptr, -1, odt_, out);
  }

  void walk_wan(Act x, void* out) {
    const vaedec_config& c = h_->cfg;
    x = conv(x, "conv_in", C3, nullptr, pick({x.buf}), sdt_);
    x = resnet(x, "mid_block.resnets.0", true, nullptr);
    x = attention(x, "mid_block.attentions.0", true);
    x = resnet(x, "mid_block.resnets.1", true, nullptr);
    for (int s = 0; s < c.n_stages && live(); ++s) {
      const std::string pre = "up_blocks." + std::to_string(s);
      Act xc;
      for (int r = 0; r < c.stage_resnets[s]; ++r) {
        const bool last = (r + 1 == c.stage_resnets[s]) && c.stage_upsample[s];
        x = resnet(x, pre + ".resnets." + std::to_string(r), true, last ? &xc : nullptr);
      }
      if (c.stage_upsample[s] == VAEDEC_UP_SPATIOTEMPORAL)
        xc = conv(xc, pre + ".upsamplers.0.time_conv", TIME, nullptr, pick({x.buf, xc.buf}), odt_);
      if (c.stage_upsample[s])
        x = conv(xc, pre + ".upsamplers.0.resample.1", UP, nullptr, pick({x.buf, xc.buf}), sdt_);
    }
    Act t = rms_norm(x, "norm_out", true, pick({x.buf}));
    conv(t, "conv_out", C3, nullptr, -1, odt_, out);
  }
};

// ---------------------------------------------------------------- create helpers
float to_f32(const vaedec_tensor& t, size_t i) {
  if (t.dtype == VAEDEC_DTYPE_F32) return static_cast<const float*>(t.data)[i];
  uint16_t u = static_cast<const uint16_t*>(t.data)[i];
  uint32_t v = static_cast<uint32_t>(u) << 16;
  float f;
  std::memcpy(&f, &v, 4);
  return f;
}

uint16_t f32_to_bf16(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7fc0;  // NaN
  u += 0x7fffu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

float bf16_to_f32(uint16_t b) {
  const uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

bool ends_with(const std::string& s, const std::string& suffix) {
  return s.size() >= suffix.size() && s.compare(s.size() - suffix.size(), suffix.size(), suffix) == 0;
}

size_t numel(const vaedec_tensor& t) {
  size_t n = 1;
  for (int i = 0; i < t.ndim; ++i) n *= (size_t)t.shape[i];
  return n;
}

// Every conv / linear / norm the architecture uses, with expected shapes.
struct Need {
  std::string name;
  int kind;                // 0 conv (weight+bias), 1 groupnorm (weight+bias), 2 rms (gamma)
  int cout, cin, kt, kh, kw;
  bool linear;             // 2D weight [cout, cin]
};

void needs_kl(const vaedec_config& c, std::vector<Need>& v) {
  auto conv = [&](const std::string& n, int ci, int co, int k) { v.push_back({n, 0, co, ci, 1, k, k, false}); };
  auto gn = [&](const std::string& n, int ch) { v.push_back({n, 1, ch, ch, 1, 1, 1, false}); };
  auto resnet = [&](const std::string& p, int ci, int co) {
    gn(p + ".norm1", ci);
    conv(p + ".conv1", ci, co, 3);
    gn(p + ".norm2", co);
    conv(p + ".conv2", co, co, 3);
    if (ci != co) conv(p + ".conv_shortcut", ci, co, 1);
  };
  const int C = c.mid_channels;
  conv("conv_in", c.latent_channels, C, 3);
  resnet("mid_block.resnets.0", C, C);
  const std::string a = "mid_block.attentions.0";
  gn(a + ".group_norm", C);
  for (const char* p : {".to_q", ".to_k", ".to_v", ".to_out.0"}) v.push_back({a + p, 0, C, C, 1, 1, 1, true});
  resnet("mid_block.resnets.1", C, C);
  int cin = C;
  for (int s = 0; s < c.n_stages; ++s) {
    const int co = c.stage_channels[s];
    for (int r = 0; r < c.stage_resnets[s]; ++r)
      resnet("up_blocks." + std::to_string(s) + ".resnets." + std::to_string(r), r == 0 ? cin : co, co);
    cin = co;
    if (c.stage_upsample[s]) {
      conv("up_blocks." + std::to_string(s) + ".upsamplers.0.conv", co, c.stage_up_channels[s], 3);
      cin = c.stage_up_channels[s];
    }
  }
  gn("conv_norm_out", cin);
  conv("conv_out", cin, c.out_channels, 3);
}

void needs_wan(const vaedec_config& c, std::vector<Need>& v) {
  auto conv3 = [&](const std::string& n, int ci, int co, int kt, int k) { v.push_back({n, 0, co, ci, kt, k, k, false}); };
  auto conv2 = [&](const std::string& n, int ci, int co, int k) { v.push_back({n, 0, co, ci, 0, k, k, false}); };
  auto rms = [&](const std::string& n, int ch) { v.push_back({n, 2, ch, ch, 1, 1, 1, false}); };
  auto resnet = [&](const std::string& p, int ci, int co) {
    rms(p + ".norm1", ci);
    conv3(p + ".conv1", ci, co, 3, 3);
    rms(p + ".norm2", co);
    conv3(p + ".conv2", co, co, 3, 3);
    if (ci != co) conv3(p + ".conv_shortcut", ci, co, 1, 1);
  };
  const int C = c.mid_channels;
  conv3("conv_in", c.latent_channels, C, 3, 3);
  resnet("mid_block.resnets.0", C, C);
  const std::string a = "mid_block.attentions.0";
  rms(a + ".norm", C);
  conv2(a + ".to_qkv", C, 3 * C, 1);
  conv2(a + ".proj", C, C, 1);
  resnet("mid_block.resnets.1", C, C);
  int cin = C;
  for (int s = 0; s < c.n_stages; ++s) {
    const int co = c.stage_channels[s];
    const std::string pre = "up_blocks." + std::to_string(s);
    for (int r = 0; r < c.stage_resnets[s]; ++r) resnet(pre + ".resnets." + std::to_string(r), r == 0 ? cin : co, co);
    cin = co;
    if (c.stage_upsample[s] == VAEDEC_UP_SPATIOTEMPORAL) v.push_back({pre + ".upsamplers.0.time_conv", 0, 2 * co, co, 3, 1, 1, false});
    if (c.stage_upsample[s]) {
      conv2(pre + ".upsamplers.0.resample.1", co, c.stage_up_channels[s], 3);
      cin = c.stage_up_channels[s];
    }
  }
  rms("norm_out", cin);
  conv3("conv_out", cin, c.out_channels, 3, 3);
}

const vaedec_tensor* find_tensor(const vaedec_tensor* ws, int n, const std::string& name) {
  for (int i = 0; i < n; ++i)
    if (ws[i].name && name == ws[i].name) return &ws[i];
  return nullptr;
}

vaedec_status upload_f32(vaedec* h, const std::vector<float>& v, float** dst, const char* what) {
  void* p = nullptr;
  vaedec_status s = h->dalloc(&p, v.size() * sizeof(float), what);
  if (s != VAEDEC_OK) return s;
  cudaError_t e = cudaMemcpy(p, v.data(), v.size() * sizeof(float), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, what);
  *dst = static_cast<float*>(p);
  return VAEDEC_OK;
}

vaedec_status validate_config(const vaedec_config* c) {
  if (c->family != VAEDEC_FAMILY_KL2D && c->family != VAEDEC_FAMILY_WAN3D) return fail(VAEDEC_ERR_INVALID_ARG, "unknown family");
  if (c->dtype != VAEDEC_DTYPE_F32 && c->dtype != VAEDEC_DTYPE_BF16) return fail(VAEDEC_ERR_INVALID_ARG, "unknown dtype");
  if (c->n_stages < 1 || c->n_stages > VAEDEC_MAX_STAGES) return fail(VAEDEC_ERR_INVALID_ARG, "n_stages out of range");
  if (c->latent_channels < 1 || c->mid_channels < 1 || c->out_channels < 1)
    return fail(VAEDEC_ERR_INVALID_ARG, "channel counts must be positive");
  for (int i = 0; i < 4; ++i)
    if (c->max_latent[i] < 1) return fail(VAEDEC_ERR_INVALID_ARG, "max_latent entries must be positive");
  if (c->family == VAEDEC_FAMILY_KL2D && c->max_latent[1] != 1) return fail(VAEDEC_ERR_INVALID_ARG, "max_latent T must be 1 for KL2D");
  std::vector<int> chans = {c->mid_channels};
  for (int s = 0; s < c->n_stages; ++s) {
    if (c->stage_channels[s] < 1 || c->stage_resnets[s] < 1 || c->stage_upsample[s] < 0 || c->stage_upsample[s] > 2)
      return fail(VAEDEC_ERR_INVALID_ARG, "bad stage description");
    if (c->stage_upsample[s] && c->stage_up_channels[s] < 1) return fail(VAEDEC_ERR_INVALID_ARG, "bad upsample channels");
    if (c->family == VAEDEC_FAMILY_KL2D && c->stage_upsample[s] == 2)
      return fail(VAEDEC_ERR_INVALID_ARG, "KL2D has no temporal upsample");
    chans.push_back(c->stage_channels[s]);
    if (c->stage_upsample[s]) chans.push_back(c->stage_up_channels[s]);
  }
  for (int ch : chans) {
    if (ch % 8 != 0) return fail(VAEDEC_ERR_UNSUPPORTED, "activation channel counts must be multiples of 8");
    if (c->dtype == VAEDEC_DTYPE_BF16 && ch % 16 != 0)
      return fail(VAEDEC_ERR_UNSUPPORTED, "bf16 path needs channel counts that are multiples of 16");
    if (ch > 2048) return fail(VAEDEC_ERR_UNSUPPORTED, "channel count too large");
    if (c->family == VAEDEC_FAMILY_KL2D && (c->norm_groups < 1 || ch % c->norm_groups != 0))
      return fail(VAEDEC_ERR_INVALID_ARG, "GroupNorm groups must divide every channel count");
    if (c->family == VAEDEC_FAMILY_WAN3D && ch > 512) return fail(VAEDEC_ERR_UNSUPPORTED, "RMSNorm supports up to 512 channels");
  }
  if (c->dtype == VAEDEC_DTYPE_BF16 && c->latent_channels % 16 != 0)
    return fail(VAEDEC_ERR_UNSUPPORTED, "bf16 path needs latent channels that are a multiple of 16");
  if (c->dtype == VAEDEC_DTYPE_BF16 && (c->mid_channels % 128 != 0 || c->mid_channels > 512))
    return fail(VAEDEC_ERR_UNSUPPORTED, "bf16 path: the fused mid-block attention needs a multiple of 128 channels, "
                                        "at most 512");
  if (c->family == VAEDEC_FAMILY_KL2D && !(c->eps > 0.f)) return fail(VAEDEC_ERR_INVALID_ARG, "eps must be positive");
  if (c->latent_patch < 0 || c->latent_patch > 2) return fail(VAEDEC_ERR_UNSUPPORTED, "latent_patch must be 0, 1 or 2");
  if (c->latent_patch == 2 && c->family != VAEDEC_FAMILY_KL2D)
    return fail(VAEDEC_ERR_INVALID_ARG, "the latent front-end is a KL2D option");
  if (c->latent_patch == 2 && !(c->latent_bn_eps > 0.f)) return fail(VAEDEC_ERR_INVALID_ARG, "latent_bn_eps must be positive");
  return VAEDEC_OK;
}

// The split axis of a request ("VAE Parallel", Strategy Selection Contract and Spatially-Sharded
// Decode): height or width as asked when that latent axis holds n_bands (one latent row or column
// per band at least); auto: the longer axis that can, width on ties.
vaedec_status resolve_band_axis(int64_t H, int64_t W, int n_bands, int axis, int* out) {
  if (n_bands < 1) return fail(VAEDEC_ERR_INVALID_ARG, "n_bands must be >= 1");
  if (axis == VAEDEC_BANDS_HEIGHT || axis == VAEDEC_BANDS_WIDTH) {
    const int64_t n = axis == VAEDEC_BANDS_HEIGHT ? H : W;
    if (n_bands > n)
      return fail(VAEDEC_ERR_INVALID_ARG, std::string("n_bands must be in [1, latent ") +
                                              (axis == VAEDEC_BANDS_HEIGHT ? "H" : "W") + "]");
    *out = axis;
    return VAEDEC_OK;
  }
  if (axis != VAEDEC_BANDS_AUTO) return fail(VAEDEC_ERR_INVALID_ARG, "unknown band axis");
  const bool w_ok = n_bands <= W, h_ok = n_bands <= H;
  if (!w_ok && !h_ok) return fail(VAEDEC_ERR_INVALID_ARG, "neither latent axis can hold n_bands bands");
  *out = (w_ok && (!h_ok || W >= H)) ? VAEDEC_BANDS_WIDTH : VAEDEC_BANDS_HEIGHT;
  return VAEDEC_OK;
}

vaedec_status check_latent(const vaedec* h, const int64_t* shape, int ndim, int n_bands, int axis = 0) {
  if (shape == nullptr) return fail(VAEDEC_ERR_INVALID_ARG, "latent shape is NULL");
  const int want = h->cfg.family == VAEDEC_FAMILY_KL2D ? 4 : 5;
  if (ndim != want) return fail(VAEDEC_ERR_INVALID_ARG, "latent ndim must be " + std::to_string(want));
  for (int i = 0; i < ndim; ++i)
    if (shape[i] < 1) return fail(VAEDEC_ERR_INVALID_ARG, "latent dims must be positive");
  if (shape[1] != (int64_t)h->cfg.latent_channels * h->patch * h->patch)
    return fail(VAEDEC_ERR_INVALID_ARG, "latent channel count mismatch");
  const int64_t B = shape[0], T = ndim == 5 ? shape[2] : 1, H = shape[ndim - 2], W = shape[ndim - 1];
  const int64_t* m = h->cfg.max_latent;
  if (B > m[0] || T > m[1] || H > m[2] || W > m[3]) return fail(VAEDEC_ERR_INVALID_ARG, "latent shape exceeds max_latent");
  // the workspace was planned for max_latent: B*T*H*W and H*W must also fit
  if (B * T * H * W > m[0] * m[1] * m[2] * m[3]) return fail(VAEDEC_ERR_INVALID_ARG, "latent shape exceeds max_latent");
  // bands split the decoder's latent grid (after the front-end's unpatchify, when there is one)
  const int64_t gh = H * h->patch, gw = W * h->patch;
  if (axis == VAEDEC_BANDS_WIDTH) {
    if (n_bands < 1 || n_bands > gw) return fail(VAEDEC_ERR_INVALID_ARG, "n_bands must be in [1, latent W]");
  } else if (n_bands < 1 || n_bands > gh) {
    return fail(VAEDEC_ERR_INVALID_ARG, "n_bands must be in [1, latent H]");
  }
  // the tensor-core attention streams keys as 16-byte-aligned rows
  if (h->dtype == kBF16 && (gh * gw) % 8 != 0)
    return fail(VAEDEC_ERR_UNSUPPORTED, "bf16 path needs latent H*W to be a multiple of 8");
  return VAEDEC_OK;
}

}  // namespace

namespace {

// Dry walk at max_latent with one band (the fp32 path's largest score buffer): the workspace slots
// with their lifetimes, the GroupNorm scratch sizes and the host-path staging sizes.
vaedec_status plan_walk(vaedec* h, Plan* plan) {
  const vaedec_config* config = &h->cfg;
  int64_t shape[5];
  int ndim;
  const int64_t* m = config->max_latent;
  if (config->family == VAEDEC_FAMILY_KL2D) {
    ndim = 4;
    shape[0] = m[0]; shape[1] = (int64_t)config->latent_channels * h->patch * h->patch; shape[2] = m[2]; shape[3] = m[3];
  } else {
    ndim = 5;
    shape[0] = m[0]; shape[1] = config->latent_channels; shape[2] = m[1]; shape[3] = m[2]; shape[4] = m[3];
  }
  Walker w(h, nullptr, true, 1);
  w.plan = plan;
  vaedec_status s = w.run(nullptr, shape, ndim, kDryOut);
  if (s != VAEDEC_OK) return s;
  int64_t oshape[5];
  if (vaedec_output_shape(h, shape, ndim, oshape) != VAEDEC_OK) return VAEDEC_ERR_INVALID_ARG;
  h->io_latent_bytes = h->es;
  h->io_out_bytes = h->es;
  for (int i = 0; i < ndim; ++i) {
    h->io_latent_bytes *= (size_t)shape[i];
    h->io_out_bytes *= (size_t)oshape[i];
  }
  return VAEDEC_OK;
}

// Places the plan's slots in one arena; returns the whole workspace in bytes (arena, GroupNorm
// chunk moments and scale/shift, host-path staging, status word).
size_t layout_workspace(vaedec* h, const Plan& plan) {
  h->arena_bytes = place_slots(plan.slots, &h->slot_off, &h->act_peak_bytes) + kArenaGuard;
  h->slot_bytes.resize(plan.slots.size());
  for (size_t i = 0; i < plan.slots.size(); ++i) h->slot_bytes[i] = plan.slots[i].bytes;
  return h->arena_bytes + std::max<size_t>(plan.part, 1) * sizeof(GnPartial) +
         2 * std::max<size_t>(plan.sc, 1) * sizeof(float) + h->io_latent_bytes + h->io_out_bytes + sizeof(int);
}

}  // namespace

void vd::record_last_error(const std::string& message) { g_err = message; }

// ====================================================================== C ABI
// Calls that launch kernels or touch the handle's device memory need the handle's device to be the
// current one: kernels launched on another device would dereference this device's pointers.
vaedec_status check_device(const vaedec* h) {
  int dev = -1;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "current device");
  if (dev != h->device)
    return fail(VAEDEC_ERR_INVALID_ARG, "the current CUDA device (" + std::to_string(dev) +
                                            ") is not the one the handle was created on (" +
                                            std::to_string(h->device) + ")");
  return VAEDEC_OK;
}

extern "C" {

const char* vaedec_last_error(void) { return g_err.c_str(); }

vaedec_status vaedec_create(const vaedec_config* config, const vaedec_tensor* weights, int n_weights,
                            vaedec_t** out) {
  g_err.clear();
  if (out == nullptr || config == nullptr) return fail(VAEDEC_ERR_INVALID_ARG, "NULL argument");
  *out = nullptr;
  if (n_weights < 0 || (n_weights > 0 && weights == nullptr)) return fail(VAEDEC_ERR_INVALID_ARG, "bad weight list");
  vaedec_status s = validate_config(config);
  if (s != VAEDEC_OK) return s;
  vaedec* h = new vaedec();
  h->cfg = *config;
  h->patch = config->latent_patch == 2 ? 2 : 1;
  h->dtype = config->dtype == VAEDEC_DTYPE_BF16 ? kBF16 : kF32;
  h->es = h->dtype == kBF16 ? 2 : 4;
  auto bail = [&](vaedec_status st) {
    delete h;
    return st;
  };
  {
    const cudaError_t e = cudaGetDevice(&h->device);
    if (e != cudaSuccess) return bail(cuda_fail(e, "current device"));
  }

  std::vector<Need> needs;
  if (config->family == VAEDEC_FAMILY_KL2D)
    needs_kl(*config, needs);
  else
    needs_wan(*config, needs);

  for (const Need& nd : needs) {
    if (nd.kind == 0) {
      const vaedec_tensor* w = find_tensor(weights, n_weights, nd.name + ".weight");
      const vaedec_tensor* b = find_tensor(weights, n_weights, nd.name + ".bias");
      if (!w || !b) return bail(fail(VAEDEC_ERR_INVALID_ARG, "missing tensor " + nd.name + ".weight/.bias"));
      // expected weight shape
      std::vector<int64_t> exp;
      if (nd.linear)
        exp = {nd.cout, nd.cin};
      else if (config->family == VAEDEC_FAMILY_WAN3D && nd.kt > 0)
        exp = {nd.cout, nd.cin, nd.kt, nd.kh, nd.kw};
      else
        exp = {nd.cout, nd.cin, nd.kh, nd.kw};
      bool okshape = w->ndim == (int)exp.size();
      for (size_t i = 0; okshape && i < exp.size(); ++i) okshape = w->shape[i] == exp[i];
      if (!okshape) return bail(fail(VAEDEC_ERR_INVALID_ARG, "unexpected shape for " + nd.name + ".weight"));
      if (b->ndim != 1 || b->shape[0] != nd.cout) return bail(fail(VAEDEC_ERR_INVALID_ARG, "unexpected shape for " + nd.name + ".bias"));
      if (w->data == nullptr || b->data == nullptr) return bail(fail(VAEDEC_ERR_INVALID_ARG, "NULL data for " + nd.name));
      const int kt = (nd.kt > 0) ? nd.kt : 1;
      const int ntaps = kt * nd.kh * nd.kw;
      DevConv dc;
      dc.cin = nd.cin;
      dc.cout = nd.cout;
      dc.ntaps = ntaps;
      dc.kt = kt;
      dc.kh = nd.kh;
      dc.kw = nd.kw;
      dc.rows = h->dtype == kBF16 ? round_up(nd.cout, 16) : nd.cout;
      // repack [cout][cin][taps] -> [rows][taps][cin]
      const size_t n = (size_t)dc.rows * ntaps * nd.cin;
      if (h->dtype == kBF16) {
        std::vector<uint16_t> buf(n, 0);
        for (int co = 0; co < nd.cout; ++co)
          for (int ci = 0; ci < nd.cin; ++ci)
            for (int t = 0; t < ntaps; ++t)
              buf[((size_t)co * ntaps + t) * nd.cin + ci] = f32_to_bf16(to_f32(*w, ((size_t)co * nd.cin + ci) * ntaps + t));
        s = h->dalloc(&dc.w, n * 2, nd.name.c_str());
        if (s != VAEDEC_OK) return bail(s);
        cudaError_t e = cudaMemcpy(dc.w, buf.data(), n * 2, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return bail(cuda_fail(e, "weight upload"));
        if (nd.cout == 3 && nd.kh == 3 && nd.kw == 3 && !nd.linear) {
          // narrow-output layout: the three kernel rows x three outputs share one 16-wide MMA N
          const size_t nn = (size_t)16 * kt * 3 * nd.cin;
          std::vector<uint16_t> wn(nn, 0);
          for (int co = 0; co < 3; ++co)
            for (int ci = 0; ci < nd.cin; ++ci)
              for (int dt = 0; dt < kt; ++dt)
                for (int i = 0; i < 3; ++i)
                  for (int j = 0; j < 3; ++j) {
                    const int t = (dt * 3 + i) * 3 + j;
                    wn[((size_t)(i * 3 + co) * (kt * 3) + dt * 3 + j) * nd.cin + ci] =
                        f32_to_bf16(to_f32(*w, ((size_t)co * nd.cin + ci) * ntaps + t));
                  }
          s = h->dalloc(&dc.wn, nn * 2, nd.name.c_str());
          if (s != VAEDEC_OK) return bail(s);
          e = cudaMemcpy(dc.wn, wn.data(), nn * 2, cudaMemcpyHostToDevice);
          if (e != cudaSuccess) return bail(cuda_fail(e, "weight upload"));
        }
        if (nd.kh == 3 && nd.kw == 3 && kt == 1 && !nd.linear &&
            (ends_with(nd.name, ".upsamplers.0.conv") || ends_with(nd.name, ".upsamplers.0.resample.1"))) {
          // the exact two-by-two phase form: per phase 7 taps, summed weights split into hi and lo
          const size_t nu = (size_t)dc.rows * 4 * kUpTaps * nd.cin;
          std::vector<uint16_t> wu(nu, 0);
          for (int ph = 0; ph < 4; ++ph) {
            UpTap tp[kUpTaps];
            up_phase_taps(ph, tp);
            for (int k = 0; k < kUpTaps; ++k)
              for (int co = 0; co < nd.cout; ++co)
                for (int ci = 0; ci < nd.cin; ++ci) {
                  double sum = 0.0;
                  for (int a = 0; a < tp[k].nrow; ++a)
                    for (int c = 0; c < tp[k].ncol; ++c) {
                      const int t = tp[k].rows[a] * 3 + tp[k].cols[c];
                      sum += bf16_to_f32(buf[((size_t)co * ntaps + t) * nd.cin + ci]);
                    }
                  const uint16_t hi = f32_to_bf16(static_cast<float>(sum));
                  const uint16_t v = tp[k].lo ? f32_to_bf16(static_cast<float>(sum - bf16_to_f32(hi))) : hi;
                  wu[((size_t)co * 4 * kUpTaps + ph * kUpTaps + k) * nd.cin + ci] = v;
                }
          }
          s = h->dalloc(&dc.wup, nu * 2, nd.name.c_str());
          if (s != VAEDEC_OK) return bail(s);
          e = cudaMemcpy(dc.wup, wu.data(), nu * 2, cudaMemcpyHostToDevice);
          if (e != cudaSuccess) return bail(cuda_fail(e, "weight upload"));
        }
      } else {
        std::vector<float> buf(n, 0.f);
        for (int co = 0; co < nd.cout; ++co)
          for (int ci = 0; ci < nd.cin; ++ci)
            for (int t = 0; t < ntaps; ++t)
              buf[((size_t)co * ntaps + t) * nd.cin + ci] = to_f32(*w, ((size_t)co * nd.cin + ci) * ntaps + t);
        s = h->dalloc(&dc.w, n * 4, nd.name.c_str());
        if (s != VAEDEC_OK) return bail(s);
        cudaError_t e = cudaMemcpy(dc.w, buf.data(), n * 4, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return bail(cuda_fail(e, "weight upload"));
      }
      std::vector<float> bias(nd.cout);
      for (int i = 0; i < nd.cout; ++i) bias[i] = to_f32(*b, i);
      s = upload_f32(h, bias, &dc.b, nd.name.c_str());
      if (s != VAEDEC_OK) return bail(s);
      h->conv[nd.name] = dc;
      static const std::string kShortcut = ".conv_shortcut";
      if (h->dtype == kBF16 && nd.name.size() > kShortcut.size() &&
          nd.name.compare(nd.name.size() - kShortcut.size(), kShortcut.size(), kShortcut) == 0) {
        // conv2 of the same block gets its bias plus this one (for the fused shortcut)
        auto c2 = h->conv.find(nd.name.substr(0, nd.name.size() - kShortcut.size()) + ".conv2");
        if (c2 != h->conv.end() && c2->second.cout == nd.cout) {
          std::vector<float> b2(nd.cout), bs(nd.cout);
          cudaError_t e = cudaMemcpy(b2.data(), c2->second.b, nd.cout * sizeof(float), cudaMemcpyDeviceToHost);
          if (e == cudaSuccess) e = cudaMemcpy(bs.data(), dc.b, nd.cout * sizeof(float), cudaMemcpyDeviceToHost);
          if (e != cudaSuccess) return bail(cuda_fail(e, "bias download"));
          for (int i = 0; i < nd.cout; ++i) b2[i] += bs[i];
          s = upload_f32(h, b2, &c2->second.b_sc, nd.name.c_str());
          if (s != VAEDEC_OK) return bail(s);
        }
      }
    } else {
      DevNorm dn;
      dn.c = nd.cout;
      const std::string gname = nd.kind == 1 ? nd.name + ".weight" : nd.name + ".gamma";
      const vaedec_tensor* g = find_tensor(weights, n_weights, gname);
      if (!g || numel(*g) != (size_t)nd.cout || !g->data)
        return bail(fail(VAEDEC_ERR_INVALID_ARG, "missing or mis-shaped " + gname));
      std::vector<float> gv(nd.cout), bv(nd.cout, 0.f);
      for (int i = 0; i < nd.cout; ++i) gv[i] = to_f32(*g, i);
      if (nd.kind == 1) {
        const vaedec_tensor* b = find_tensor(weights, n_weights, nd.name + ".bias");
        if (!b || numel(*b) != (size_t)nd.cout || !b->data)
          return bail(fail(VAEDEC_ERR_INVALID_ARG, "missing or mis-shaped " + nd.name + ".bias"));
        for (int i = 0; i < nd.cout; ++i) bv[i] = to_f32(*b, i);
      }
      s = upload_f32(h, gv, &dn.g, gname.c_str());
      if (s != VAEDEC_OK) return bail(s);
      s = upload_f32(h, bv, &dn.b, gname.c_str());
      if (s != VAEDEC_OK) return bail(s);
      h->norm[nd.name] = dn;
    }
  }

  if (h->patch > 1) {
    // inverse latent BatchNorm of the front-end: per patched channel scale = sqrt(var + eps), shift = mean
    const int cp = config->latent_channels * h->patch * h->patch;
    const vaedec_tensor* mt = find_tensor(weights, n_weights, "bn.running_mean");
    const vaedec_tensor* vt = find_tensor(weights, n_weights, "bn.running_var");
    if (!mt || !vt || mt->ndim != 1 || vt->ndim != 1 || mt->shape[0] != cp || vt->shape[0] != cp ||
        mt->data == nullptr || vt->data == nullptr)
      return bail(fail(VAEDEC_ERR_INVALID_ARG, "missing or mis-shaped bn.running_mean / bn.running_var"));
    std::vector<float> sc(cp), sh(cp);
    for (int i = 0; i < cp; ++i) {
      const float var = to_f32(*vt, i);
      if (!(var + config->latent_bn_eps > 0.f)) return bail(fail(VAEDEC_ERR_INVALID_ARG, "bn.running_var + eps must be positive"));
      sc[i] = std::sqrt(var + config->latent_bn_eps);
      sh[i] = to_f32(*mt, i);
    }
    void* tmp = nullptr;
    s = h->dalloc(&tmp, cp * sizeof(float), "latent batchnorm scale");
    if (s != VAEDEC_OK) return bail(s);
    h->bn_scale = static_cast<float*>(tmp);
    s = h->dalloc(&tmp, cp * sizeof(float), "latent batchnorm shift");
    if (s != VAEDEC_OK) return bail(s);
    h->bn_shift = static_cast<float*>(tmp);
    cudaError_t e = cudaMemcpy(h->bn_scale, sc.data(), cp * sizeof(float), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(h->bn_shift, sh.data(), cp * sizeof(float), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return bail(cuda_fail(e, "latent batchnorm upload"));
  }

  Plan plan;
  s = plan_walk(h, &plan);
  if (s != VAEDEC_OK) return bail(s);
  h->ws_bytes = layout_workspace(h, plan);
  s = h->dalloc(&h->arena, h->arena_bytes, "workspace arena");
  void* tmp = nullptr;
  if (s == VAEDEC_OK) s = h->dalloc(&tmp, std::max<size_t>(plan.part, 1) * sizeof(GnPartial), "groupnorm partials");
  h->gn_part = static_cast<GnPartial*>(tmp);
  if (s == VAEDEC_OK) s = h->dalloc(&tmp, std::max<size_t>(plan.sc, 1) * sizeof(float), "groupnorm scale");
  h->gn_scale = static_cast<float*>(tmp);
  if (s == VAEDEC_OK) s = h->dalloc(&tmp, std::max<size_t>(plan.sc, 1) * sizeof(float), "groupnorm shift");
  h->gn_shift = static_cast<float*>(tmp);
  if (s == VAEDEC_OK) s = h->dalloc(&h->io_latent, h->io_latent_bytes, "host-path latent");
  if (s == VAEDEC_OK) s = h->dalloc(&h->io_out, h->io_out_bytes, "host-path output");
  if (s == VAEDEC_OK) s = h->dalloc(&tmp, sizeof(int), "status word");
  h->status = static_cast<int*>(tmp);
  if (s != VAEDEC_OK) return bail(s);
  cudaError_t e = cudaMemset(h->status, 0, sizeof(int));
  if (e != cudaSuccess) return bail(cuda_fail(e, "status init"));
  *out = h;
  return VAEDEC_OK;
}

void vaedec_destroy(vaedec_t* h) {
  if (h == nullptr) return;
  // the handle's memory is freed on its own device; the caller's current device is restored
  const int hd = h->device;
  int cur = -1;
  const bool other = cudaGetDevice(&cur) == cudaSuccess && cur != hd;
  if (other) cudaSetDevice(hd);
  cudaDeviceSynchronize();
  delete h;
  if (other) cudaSetDevice(cur);
}

vaedec_status vaedec_output_shape(const vaedec_t* h, const int64_t* shape, int ndim, int64_t* out_shape) {
  if (h == nullptr || shape == nullptr || out_shape == nullptr) return fail(VAEDEC_ERR_INVALID_ARG, "NULL argument");
  const int want = h->cfg.family == VAEDEC_FAMILY_KL2D ? 4 : 5;
  if (ndim != want) return fail(VAEDEC_ERR_INVALID_ARG, "latent ndim must be " + std::to_string(want));
  int64_t f = 1, T = ndim == 5 ? shape[2] : 1;
  for (int s = 0; s < h->cfg.n_stages; ++s) {
    if (h->cfg.stage_upsample[s]) f *= 2;
    if (h->cfg.stage_upsample[s] == VAEDEC_UP_SPATIOTEMPORAL) T = 2 * T - 1;
  }
  f *= h->patch;   // the front-end's unpatchify (KL2D with a patched latent)
  out_shape[0] = shape[0];
  out_shape[1] = h->cfg.out_channels;
  if (ndim == 5) {
    out_shape[2] = T;
    out_shape[3] = shape[3] * f;
    out_shape[4] = shape[4] * f;
  } else {
    out_shape[2] = shape[2] * f;
    out_shape[3] = shape[3] * f;
  }
  return VAEDEC_OK;
}

vaedec_status vaedec_plan_workspace(const vaedec_config* config, size_t* bytes, size_t* arena_bytes,
                                    size_t* peak_live_bytes) {
  g_err.clear();
  if (config == nullptr || bytes == nullptr) return fail(VAEDEC_ERR_INVALID_ARG, "NULL argument");
  vaedec_status s = validate_config(config);
  if (s != VAEDEC_OK) return s;
  vaedec h;   // layer shapes only: no weights, no device memory
  h.cfg = *config;
  h.patch = config->latent_patch == 2 ? 2 : 1;
  h.dtype = config->dtype == VAEDEC_DTYPE_BF16 ? kBF16 : kF32;
  h.es = h.dtype == kBF16 ? 2 : 4;
  std::vector<Need> needs;
  if (config->family == VAEDEC_FAMILY_KL2D)
    needs_kl(*config, needs);
  else
    needs_wan(*config, needs);
  for (const Need& nd : needs) {
    if (nd.kind == 0) {
      DevConv dc;
      dc.cin = nd.cin;
      dc.cout = nd.cout;
      dc.kt = nd.kt > 0 ? nd.kt : 1;
      dc.kh = nd.kh;
      dc.kw = nd.kw;
      dc.ntaps = dc.kt * nd.kh * nd.kw;
      dc.rows = h.dtype == kBF16 ? round_up(nd.cout, 16) : nd.cout;
      h.conv[nd.name] = dc;
    } else {
      DevNorm dn;
      dn.c = nd.cout;
      h.norm[nd.name] = dn;
    }
  }
  if (h.dtype == kBF16) {
    // as at create: a block with a 1x1 shortcut gets a combined conv2 bias (never read by a dry walk)
    static const std::string kShortcut = ".conv_shortcut";
    for (auto& kv : h.conv) {
      const std::string& nm = kv.first;
      if (nm.size() <= kShortcut.size() || nm.compare(nm.size() - kShortcut.size(), kShortcut.size(), kShortcut) != 0)
        continue;
      auto c2 = h.conv.find(nm.substr(0, nm.size() - kShortcut.size()) + ".conv2");
      if (c2 != h.conv.end() && c2->second.cout == kv.second.cout) c2->second.b_sc = reinterpret_cast<float*>(kDryOut);
    }
  }
  Plan plan;
  s = plan_walk(&h, &plan);
  if (s != VAEDEC_OK) return s;
  *bytes = layout_workspace(&h, plan);
  {
    // the layout covers a decode walk at max_latent (same slots, same sizes)
    const int64_t* m = config->max_latent;
    int64_t shape[5];
    int ndim;
    if (config->family == VAEDEC_FAMILY_KL2D) {
      ndim = 4;
      shape[0] = m[0]; shape[1] = (int64_t)config->latent_channels * h.patch * h.patch; shape[2] = m[2]; shape[3] = m[3];
    } else {
      ndim = 5;
      shape[0] = m[0]; shape[1] = config->latent_channels; shape[2] = m[1]; shape[3] = m[2]; shape[4] = m[3];
    }
    Walker w(&h, nullptr, true, 1);
    s = w.run(nullptr, shape, ndim, kDryOut);
    if (s != VAEDEC_OK) return s;
  }
  if (arena_bytes) *arena_bytes = h.arena_bytes;
  if (peak_live_bytes) *peak_live_bytes = h.act_peak_bytes;
  return VAEDEC_OK;
}

vaedec_status vaedec_workspace_bytes(const vaedec_t* h, size_t* bytes) {
  if (h == nullptr || bytes == nullptr) return fail(VAEDEC_ERR_INVALID_ARG, "NULL argument");
  *bytes = h->ws_bytes;
  return VAEDEC_OK;
}

vaedec_status vaedec_decode(vaedec_t* h, const void* latent, const int64_t* shape, int ndim, void* out, int n_bands,
                            void* stream) {
  if (h == nullptr || latent == nullptr || out == nullptr) return fail(VAEDEC_ERR_INVALID_ARG, "NULL argument");
  vaedec_status s = check_device(h);
  if (s != VAEDEC_OK) return s;
  s = check_latent(h, shape, ndim, n_bands);
  if (s != VAEDEC_OK) return s;
  Walker w(h, static_cast<cudaStream_t>(stream), false, n_bands);
  return w.run(latent, shape, ndim, out);
}

vaedec_status vaedec_band_axis(const int64_t* latent_shape, int ndim, int n_bands, int axis, int* axis_out) {
  if (latent_shape == nullptr || axis_out == nullptr) return fail(VAEDEC_ERR_INVALID_ARG, "NULL argument");
  if (ndim != 4 && ndim != 5) return fail(VAEDEC_ERR_INVALID_ARG, "latent ndim must be 4 or 5");
  return resolve_band_axis(latent_shape[ndim - 2], latent_shape[ndim - 1], n_bands, axis, axis_out);
}

vaedec_status vaedec_decode_bands(vaedec_t* h, const void* latent, const int64_t* shape, int ndim, void* out,
                                  int n_bands, int axis, void* stream) {
  if (h == nullptr || latent == nullptr || out == nullptr || shape == nullptr)
    return fail(VAEDEC_ERR_INVALID_ARG, "NULL argument");
  if (ndim != 4 && ndim != 5) return fail(VAEDEC_ERR_INVALID_ARG, "latent ndim must be 4 or 5");
  int ax = 0;
  vaedec_status s = check_device(h);
  if (s != VAEDEC_OK) return s;
  s = resolve_band_axis(shape[ndim - 2] * h->patch, shape[ndim - 1] * h->patch, n_bands, axis, &ax);
  if (s != VAEDEC_OK) return s;
  s = check_latent(h, shape, ndim, n_bands, ax);
  if (s != VAEDEC_OK) return s;
  Walker w(h, static_cast<cudaStream_t>(stream), false, n_bands, ax);
  return w.run(latent, shape, ndim, out);
}

vaedec_status vaedec_sync(vaedec_t* h, void* stream) {
  if (h == nullptr) return fail(VAEDEC_ERR_INVALID_ARG, "NULL handle");
  vaedec_status s = check_device(h);
  if (s != VAEDEC_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  int word = 0;
  e = cudaMemcpy(&word, h->status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  if (word != 0) {
    cudaMemset(h->status, 0, sizeof(int));
    return fail(VAEDEC_ERR_TIMEOUT, "a kernel's bounded wait ran out (status word " + std::to_string(word) + ")");
  }
  return VAEDEC_OK;
}

vaedec_status vaedec_decode_host(vaedec_t* h, const void* latent_host, const int64_t* shape, int ndim, void* out_host,
                                 int n_bands, void* stream) {
  if (h == nullptr || latent_host == nullptr || out_host == nullptr) return fail(VAEDEC_ERR_INVALID_ARG, "NULL argument");
  vaedec_status s = check_device(h);
  if (s != VAEDEC_OK) return s;
  s = check_latent(h, shape, ndim, n_bands);
  if (s != VAEDEC_OK) return s;
  int64_t oshape[5];
  s = vaedec_output_shape(h, shape, ndim, oshape);
  if (s != VAEDEC_OK) return s;
  size_t in_b = h->es, out_b = h->es;
  for (int i = 0; i < ndim; ++i) {
    in_b *= (size_t)shape[i];
    out_b *= (size_t)oshape[i];
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(h->io_latent, latent_host, in_b, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return cuda_fail(e, "latent upload");
  s = vaedec_decode(h, h->io_latent, shape, ndim, h->io_out, n_bands, stream);
  if (s != VAEDEC_OK) return s;
  e = cudaMemcpyAsync(out_host, h->io_out, out_b, cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return cuda_fail(e, "output download");
  return vaedec_sync(h, stream);
}

vaedec_status vaedec_band_attention_work_bytes(int F, int grid_h, int grid_w, int C, size_t* bytes) {
  if (bytes == nullptr) return fail(VAEDEC_ERR_INVALID_ARG, "NULL argument");
  if (F < 1 || grid_h < 1 || grid_w < 1 || C < 1) return fail(VAEDEC_ERR_INVALID_ARG, "sizes must be positive");
  *bytes = flash_work_bytes(F, (long long)grid_h * grid_w, C);
  return VAEDEC_OK;
}

vaedec_status vaedec_band_attention(const void* q, const void* k, const void* vt, void* o, int F, int grid_h,
                                    int grid_w, int C, int n_bands, void* work, size_t work_bytes, int* status,
                                    void* stream) {
  if (q == nullptr || k == nullptr || vt == nullptr || o == nullptr || status == nullptr)
    return fail(VAEDEC_ERR_INVALID_ARG, "NULL argument");
  if (F < 1 || grid_h < 1 || grid_w < 1) return fail(VAEDEC_ERR_INVALID_ARG, "sizes must be positive");
  if (C < 128 || C > 512 || C % 128 != 0) return fail(VAEDEC_ERR_INVALID_ARG, "C must be a multiple of 128, at most 512");
  const long long ntok = (long long)grid_h * grid_w;
  if (ntok % 8 != 0) return fail(VAEDEC_ERR_INVALID_ARG, "grid_h * grid_w must be a multiple of 8");
  if (n_bands < 1 || n_bands > grid_h) return fail(VAEDEC_ERR_INVALID_ARG, "n_bands must be in [1, grid_h]");
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(vt) |
       reinterpret_cast<uintptr_t>(o) | reinterpret_cast<uintptr_t>(work)) & 15)
    return fail(VAEDEC_ERR_INVALID_ARG, "device pointers must be 16-byte aligned");
  const size_t need = flash_work_bytes(F, ntok, C);
  if (need > 0 && (work == nullptr || work_bytes < need))
    return fail(VAEDEC_ERR_INVALID_ARG, "work buffer smaller than vaedec_band_attention_work_bytes (" +
                                            std::to_string(need) + " bytes)");
  FlashArgs fa;
  fa.q = q;
  fa.k = k;
  fa.vt = vt;
  fa.out = o;
  fa.part = static_cast<float*>(work);
  fa.ml = need > 0 ? static_cast<char*>(work) + (size_t)flash_splits(ntok) * (size_t)F * (size_t)ntok * C * sizeof(float)
                   : nullptr;
  fa.F = F;
  fa.ntok = ntok;
  fa.C = C;
  fa.U = grid_w;
  fa.n_seg = n_bands;
  fa.seg_q = grid_h / n_bands;
  fa.seg_rem = grid_h % n_bands;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const char* why = nullptr;
  cudaError_t e = launch_attn_flash(fa, status, st, &why);
  if (e == cudaSuccess) e = launch_attn_combine(fa, st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(why ? VAEDEC_ERR_INVALID_ARG : VAEDEC_ERR_CUDA,
                std::string("band attention: ") + (why ? why : cudaGetErrorString(e)));
  }
  return VAEDEC_OK;
}

vaedec_status vaedec_debug_inject_fault(int kind, int nth) {
  if (kind < 0 || kind > 2 || (kind != 0 && nth < 1)) return fail(VAEDEC_ERR_INVALID_ARG, "bad fault kind or count");
  g_fault_kind.store(0);
  g_fault_left.store(nth);
  g_fault_kind.store(kind);
  return VAEDEC_OK;
}

vaedec_status vaedec_debug_set_wait_limit(uint64_t ns) {
  cudaError_t e = set_wait_limit_conv_tc(ns);
  if (e == cudaSuccess) e = set_wait_limit_conv_halo(ns);
  if (e == cudaSuccess) e = set_wait_limit_conv_halo_t(ns);
  if (e == cudaSuccess) e = set_wait_limit_conv_narrow(ns);
  if (e == cudaSuccess) e = set_wait_limit_gemm_cm(ns);
  if (e == cudaSuccess) e = set_wait_limit_attn_flash(ns);
  if (e != cudaSuccess) return fail(VAEDEC_ERR_CUDA, std::string("setting the wait limit: ") + cudaGetErrorString(e));
  return VAEDEC_OK;
}

vaedec_status vaedec_debug_wait_probe(vaedec_t* h, void* stream) {
  if (h == nullptr) return fail(VAEDEC_ERR_INVALID_ARG, "NULL handle");
  const vaedec_status s = check_device(h);
  if (s != VAEDEC_OK) return s;
  cudaError_t e = launch_wait_probe(h->status, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(VAEDEC_ERR_CUDA, std::string("wait probe: ") + cudaGetErrorString(e));
  return VAEDEC_OK;
}

vaedec_status vaedec_launch_count(const vaedec_t* h, uint64_t* n) {
  if (h == nullptr || n == nullptr) return fail(VAEDEC_ERR_INVALID_ARG, "NULL argument");
  *n = h->launches;
  return VAEDEC_OK;
}

vaedec_status vaedec_profile_enable(vaedec_t* h, int enable) {
  if (h == nullptr) return fail(VAEDEC_ERR_INVALID_ARG, "NULL handle");
  h->profile = enable != 0;
  h->prof_ops = 0;
  return VAEDEC_OK;
}

vaedec_status vaedec_profile_read(vaedec_t* h, float* ms, int max_ops, int* n_ops) {
  if (h == nullptr || n_ops == nullptr || (ms == nullptr && max_ops > 0)) return fail(VAEDEC_ERR_INVALID_ARG, "NULL argument");
  const vaedec_status s = check_device(h);
  if (s != VAEDEC_OK) return s;
  *n_ops = h->prof_ops;
  for (int i = 0; i < h->prof_ops && i < max_ops; ++i) {
    cudaError_t e = cudaEventSynchronize(h->prof_ev[2 * i + 1]);
    if (e != cudaSuccess) return cuda_fail(e, "profile event synchronize");
    e = cudaEventElapsedTime(&ms[i], h->prof_ev[2 * i], h->prof_ev[2 * i + 1]);
    if (e != cudaSuccess) return cuda_fail(e, "profile event elapsed");
  }
  return VAEDEC_OK;
}

vaedec_status vaedec_debug_num_ops(vaedec_t* h, const int64_t* shape, int ndim, int n_bands, int* n_ops) {
  if (h == nullptr || n_ops == nullptr) return fail(VAEDEC_ERR_INVALID_ARG, "NULL argument");
  vaedec_status s = check_latent(h, shape, ndim, n_bands);
  if (s != VAEDEC_OK) return s;
  Walker w(h, nullptr, true, n_bands);
  s = w.run(nullptr, shape, ndim, kDryOut);
  *n_ops = w.n_ops;
  return s;
}

vaedec_status vaedec_debug_op_desc(vaedec_t* h, const int64_t* shape, int ndim, int n_bands, int op, char* buf,
                                   int buf_len) {
  if (h == nullptr || buf == nullptr || buf_len < 1) return fail(VAEDEC_ERR_INVALID_ARG, "NULL argument");
  vaedec_status s = check_latent(h, shape, ndim, n_bands);
  if (s != VAEDEC_OK) return s;
  std::string d;
  Walker w(h, nullptr, true, n_bands);
  w.stop_at = op;
  w.desc_out = &d;
  s = w.run(nullptr, shape, ndim, kDryOut);
  if (s != VAEDEC_OK) return s;
  if (d.empty()) return fail(VAEDEC_ERR_INVALID_ARG, "op index out of range");
  if ((int)d.size() + 1 > buf_len) return fail(VAEDEC_ERR_INVALID_ARG, "description buffer too small");
  std::memcpy(buf, d.c_str(), d.size() + 1);
  return VAEDEC_OK;
}

vaedec_status vaedec_debug_run_until(vaedec_t* h, const void* latent, const int64_t* shape, int ndim, int n_bands,
                                     int op, void* dst_in, size_t in_bytes, void* dst_aux, size_t aux_bytes,
                                     void* dst_out, size_t out_bytes, void* stream) {
  if (h == nullptr || latent == nullptr) return fail(VAEDEC_ERR_INVALID_ARG, "NULL argument");
  vaedec_status s = check_device(h);
  if (s != VAEDEC_OK) return s;
  s = check_latent(h, shape, ndim, n_bands);
  if (s != VAEDEC_OK) return s;
  if (op < 0) return fail(VAEDEC_ERR_INVALID_ARG, "op index out of range");
  // the final op writes the caller's output: route it to a scratch output buffer
  Walker w(h, static_cast<cudaStream_t>(stream), false, n_bands);
  w.stop_at = op;
  w.d_in = dst_in;
  w.in_b = in_bytes;
  w.d_aux = dst_aux;
  w.aux_b = aux_bytes;
  w.d_out = dst_out;
  w.out_b = out_bytes;
  s = w.run(latent, shape, ndim, h->io_out);
  if (s != VAEDEC_OK) return s;
  if (!w.stopped) return fail(VAEDEC_ERR_INVALID_ARG, "op index out of range");
  return vaedec_sync(h, stream);
}

}  // extern "C"
